// Host-side interface between the C-ABI facade (api.cu) and the kernel
// translation units.  Plain structs passed by value to the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

#include <string>
#include <utility>

namespace dsa {

struct SeqArgs {
  int32_t B, T, max_ctx, q_per_seq;
  const int32_t* q_seq;
  const int32_t* q_pos;
  const int32_t* block_table;
  int32_t bt_stride, page_size;
  int64_t cache_rows;
  int64_t n_pages;  // cache_rows / page_size
};

struct IndexerArgs {
  int32_t H_I, D_I;
  bool e4m3;  // e4m3 codes (else fp32 values)
  bool mx;    // e4m3 codes with E8M0 scales per 32 elements (q_scale/k_scale uint8)
  const void* q;
  const void* q_scale;  // fp32 [T, H_I] (may be null) or uint8 [T, H_I, D_I/32] (mx)
  const float* w;
  const void* k;
  const void* k_scale;  // fp32 [rows] (may be null) or uint8 [rows, D_I/32] (mx)
  float* scores;
  int64_t ld;
};

enum class MlaKind { kF32 = 0, kBF16 = 1, kFP8Row = 2, kFP8Tile = 3 };   // kFP8Tile: scale per 128 latent dims

struct MlaArgs {
  int32_t H, d_latent, d_rope;
  MlaKind kind;
  const void* q;
  const void* kv;
  int64_t row_bytes;
  float softmax_scale;
  const int32_t* idx;
  int32_t K;
  void* out;
  float* lse;  // may be null
};

struct LaunchEnv {
  cudaStream_t stream;
  int num_sms;
  int device;
};

// Each launcher validates kernel-specific limits, enqueues its kernels and
// appends a short description of what it launched to *plan.  Returns
// cudaSuccess or the launch error; `unsupported` is set (and nothing launched)
// when no kernel covers the arguments.

// Lightning indexer.
cudaError_t launch_indexer(const SeqArgs& seq, const IndexerArgs& a, const LaunchEnv& env,
                           std::string* plan, bool* unsupported, std::string* why);

// Fused decode plan: indexer scores kept in shared memory and the Top-K selected
// in the same kernel (clusters of CTAs per query); writes idx [T, K] only.  Sets
// *unsupported (and launches nothing) when the arguments call for the chained plan.
cudaError_t launch_decode_fused(const SeqArgs& seq, const IndexerArgs& a, int32_t K, int32_t* idx,
                                const LaunchEnv& env, std::string* plan, bool* unsupported, std::string* why);

// Top-K.
cudaError_t launch_topk(const SeqArgs& seq, const float* scores, int64_t ld, int32_t K,
                        int32_t* idx, const LaunchEnv& env, std::string* plan);

// Sparse MLA attention.  workspace may be null (ws_bytes 0).
size_t attn_workspace_bytes(const SeqArgs& seq, const MlaArgs& a, int num_sms);
cudaError_t launch_attn(const SeqArgs& seq, const MlaArgs& a, void* workspace, size_t ws_bytes,
                        const LaunchEnv& env, std::string* plan, bool* unsupported,
                        std::string* why);

// Launches a kernel, when `pdl` with programmatic stream serialization (it
// may launch while the previous kernel on the stream is finishing; every
// kernel of this library waits for its predecessor with griddepcontrol.wait
// before reading anything), and when cluster > 1 as clusters of `cluster` CTAs
// along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The indexer prolog (projections, key normalisation, quantisation, key append).
struct PrologArgs {
  int32_t d_model, d_q, H_I;
  const void* x;        // bf16 [T, d_model]
  const void* x_q;      // bf16 [T, d_q]
  const void* w_q;      // bf16 [H_I * 128, d_q]
  const void* w_k;      // bf16 [128, d_model]
  const void* w_w;      // bf16 [H_I, d_model]
  const float* gamma;   // [128]
  const float* beta;    // [128]
  uint8_t* q_codes;     // [T, H_I, 128]
  float* q_scale;       // [T, H_I]
  float* w;             // [T, H_I]
  uint8_t* k_cache;     // [cache_rows, 128]
  float* k_scale;       // [cache_rows]
};
size_t prolog_workspace_bytes(int T, int H_I, int d_model, int d_q, int num_sms);
cudaError_t launch_prolog(const SeqArgs& seq, const PrologArgs& a, void* workspace, const LaunchEnv& env,
                          std::string* plan, bool* unsupported, std::string* why);

// Cache writers (the new tokens' index keys / latent rows into the paged caches).
cudaError_t launch_index_append(const SeqArgs& seq, int32_t D, bool bf16_in, const void* k_new, uint8_t* k_cache,
                                float* k_scale, const LaunchEnv& env, std::string* plan);
cudaError_t launch_index_append_mx(const SeqArgs& seq, int32_t D, bool bf16_in, const void* k_new, uint8_t* k_cache,
                                   uint8_t* k_exp, const LaunchEnv& env, std::string* plan);
cudaError_t launch_latent_append(const SeqArgs& seq, const MlaArgs& a, const void* kv_new, void* kv_cache,
                                 const LaunchEnv& env, std::string* plan);

// Sets the text dsa_last_error() returns on the calling thread.
void set_last_error(const std::string& msg);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on `device` (which
// must be current), once per (kernel, device); later calls return the first
// call's result.  Thread-safe.
cudaError_t ensure_smem_limit(const void* kernel, int bytes, int device);
// Whether one cluster of `cl` CTAs of `kernel` (`threads` threads, `smem` bytes of
// dynamic shared memory each) can be resident on `device`; the occupancy query is
// made once per distinct argument set (and allows non-portable sizes above 8).
bool cluster_fits(const void* kernel, int device, int cl, int threads, size_t smem);

// The failure-detection testing aid (dsa_debug_withhold_arrival): the wait
// bound the kernels use and whether the attention producer withholds an arrival.
void debug_wait_state(uint64_t* wait_limit_ns, uint32_t* withhold);

// Scratch bytes dsa_decode_step needs for these descriptors on the current
// device, with the status (and dsa_last_error text) dsa_decode_step itself
// would return for a bad descriptor.
dsa_status_t decode_workspace_need(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, int32_t K, size_t* need);

// Tensor-map encoder (driver entry point, resolved once).
bool encode_tmap_2d_u8(void* tmap_out, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       std::string* why);
// Same for 1- or 2-byte elements (inner / box_inner counted in elements), 128-byte swizzle.
bool encode_tmap_2d(void* tmap_out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, std::string* why);

}  // namespace dsa

// Per-translation-unit device status words (read and clear; 0xFFFFFFFF on error).
uint32_t dsa_status_read_clear_indexer();
uint32_t dsa_status_read_clear_topk();
uint32_t dsa_status_read_clear_attn();
uint32_t dsa_status_read_clear_cache();
uint32_t dsa_status_read_clear_prolog();
