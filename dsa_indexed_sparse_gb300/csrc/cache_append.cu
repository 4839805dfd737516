// Cache writers: the new tokens' indexer keys and latent rows into the paged
// caches (the prolog side of the step).
//
// "Large Language Model Inference Acceleration in Practice", section 3.2 (the
// indexer prolog normalises K and updates the key cache) and section 4
// (layered quantisation: FP8 index keys and KV cache); "Day0 Inference
// Adaptation and Performance Optimization for Kimi K3.1 Pro", section 4.  The
// formats written are the ones the scoring and attention kernels read:
//  * index keys: uint8 [cache_rows, D] e4m3 codes + fp32 [cache_rows] scales,
//    scale = amax / 448 (1 for an all-zero vector), code = the E4M3 value
//    nearest to x / scale (ties to even, saturated to +-448), both divisions
//    IEEE round-to-nearest in fp32;
//  * index keys, MXFP8: uint8 codes + uint8 [cache_rows, D/32] E8M0 bytes; block
//    b of 32 elements gets exponent floor(log2 amax_b) - 8 (-127 for an all-zero
//    block), code = the E4M3 value nearest to x * 2^-exponent (exact power-of-two
//    quotient; ties to even, saturated to +-448);
//  * latent rows: bf16 or fp32 rows copied; 656-byte FP8 rows built as
//    [512 e4m3 codes of the latent part][fp32 scale][12 zero bytes][64 bf16 rope],
//    or with one power-of-two scale per 128 latent dims (the same exponent rule
//    on 128-element tiles) as [512 codes][4 fp32 scales][64 bf16 rope].
// One warp per new token; the token goes to the cache row of its position
// q_pos[t] in sequence q_seq[t] through the page table.  Positions must be
// distinct within a call (two tokens on one row race).
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdio>

#include "dsa_device.cuh"
#include "dsa_internal.h"

DSA_DEFINE_STATUS_WORD(cache)

namespace dsa {
namespace {

constexpr int kAppendWarps = 8;
constexpr int kMaxChunks = 8;   // 4-element chunks per lane: D <= 1024

__device__ __forceinline__ uint32_t e4m3_code(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Cache row of new token t, or -1 (flagged) when its position or page is invalid.
__device__ __forceinline__ int64_t append_row(const SeqArgs& seq, int t) {
  const int qp = __ldg(seq.q_pos + t), b = __ldg(seq.q_seq + t);
  if (qp < 0 || qp >= seq.max_ctx || b < 0 || b >= seq.B) {
    atomicOr(&g_status_cache, kDevBadPos);
    return -1;
  }
  return phys_row(seq.block_table + static_cast<int64_t>(b) * seq.bt_stride, qp, seq.page_size, seq.n_pages,
                  &g_status_cache);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <bool kBf16In>
__global__ void __launch_bounds__(kAppendWarps * 32)
    index_append_kernel(SeqArgs seq, int32_t D, const void* k_new, uint8_t* k_cache, float* k_scale) {
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= seq.T) return;
  const int64_t row = append_row(seq, t);
  if (row < 0) return;
  const int nq = D / 4;
  float v[kMaxChunks][4];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = lane + 32 * k;
    if (c < nq) {
      if (kBf16In) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(k_new) +
                                                             static_cast<int64_t>(t) * D) + c);
        v[k][0] = bf16_bits_to_float(u.x & 0xFFFFu);
        v[k][1] = bf16_bits_to_float(u.x >> 16);
        v[k][2] = bf16_bits_to_float(u.y & 0xFFFFu);
        v[k][3] = bf16_bits_to_float(u.y >> 16);
      } else {
        const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(k_new) +
                                                               static_cast<int64_t>(t) * D) + c);
        v[k][0] = f.x;
        v[k][1] = f.y;
        v[k][2] = f.z;
        v[k][3] = f.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(v[k][i]));
    }
  }
  amax = warp_max(amax);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t* dst = reinterpret_cast<uint32_t*>(k_cache + row * D);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = lane + 32 * k;
    if (c < nq)
      dst[c] = e4m3_code(__fdiv_rn(v[k][0], scale)) | (e4m3_code(__fdiv_rn(v[k][1], scale)) << 8) |
               (e4m3_code(__fdiv_rn(v[k][2], scale)) << 16) | (e4m3_code(__fdiv_rn(v[k][3], scale)) << 24);
  }
  if (lane == 0) k_scale[row] = scale;
}

// MX shared exponent of a block whose largest magnitude is amax: floor(log2 amax)
// - 8 (8: exponent of E4M3's largest normal), clamped to [-127, 127]; -127 for 0.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  return max(-127, min(127, ilogbf(amax) - 8));
}

// MXFP8 index keys: blocks of 32 elements are 8 consecutive lanes' 4-element
// chunks (chunk c = lane + 32 k), so a block's amax is a 3-step shuffle max.
template <bool kBf16In>
__global__ void __launch_bounds__(kAppendWarps * 32)
    index_append_mx_kernel(SeqArgs seq, int32_t D, const void* k_new, uint8_t* k_cache, uint8_t* k_exp) {
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= seq.T) return;
  const int64_t row = append_row(seq, t);
  if (row < 0) return;
  const int nq = D / 4;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = lane + 32 * k;
    if (32 * k >= nq) break;        // warp-uniform: nq is a multiple of 8
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (c < nq) {
      if (kBf16In) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(k_new) +
                                                             static_cast<int64_t>(t) * D) + c);
        v[0] = bf16_bits_to_float(u.x & 0xFFFFu);
        v[1] = bf16_bits_to_float(u.x >> 16);
        v[2] = bf16_bits_to_float(u.y & 0xFFFFu);
        v[3] = bf16_bits_to_float(u.y >> 16);
      } else {
        const float4 f = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(k_new) +
                                                               static_cast<int64_t>(t) * D) + c);
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
      }
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = mx_exponent(amax);
    if (c < nq) {
      reinterpret_cast<uint32_t*>(k_cache + row * D)[c] =
          e4m3_code(ldexpf(v[0], -e)) | (e4m3_code(ldexpf(v[1], -e)) << 8) |
          (e4m3_code(ldexpf(v[2], -e)) << 16) | (e4m3_code(ldexpf(v[3], -e)) << 24);
      if ((lane & 7) == 0) k_exp[row * (D / 32) + c / 8] = static_cast<uint8_t>(e + 127);
    }
  }
}

// bf16 / fp32 rows: a 16-byte-vector copy of row_in bytes.
__global__ void __launch_bounds__(kAppendWarps * 32)
    latent_copy_kernel(SeqArgs seq, int64_t row_in, int64_t row_bytes, const void* kv_new, uint8_t* cache) {
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= seq.T) return;
  const int64_t row = append_row(seq, t);
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(kv_new) + t * row_in);
  uint4* dst = reinterpret_cast<uint4*>(cache + row * row_bytes);
  for (int64_t c = lane; c < row_in / 16; c += 32) dst[c] = __ldg(src + c);
}

// 656-byte FP8 rows from bf16 [576] input rows (512 latent + 64 rope).
__global__ void __launch_bounds__(kAppendWarps * 32)
    latent_fp8_kernel(SeqArgs seq, int64_t row_bytes, const uint16_t* kv_new, uint8_t* cache) {
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= seq.T) return;
  const int64_t row = append_row(seq, t);
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(kv_new + static_cast<int64_t>(t) * 576);
  uint8_t* dst = cache + row * row_bytes;
  // latent values [16 lane, 16 lane + 16)
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 u = __ldg(src + 2 * lane + h);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * h + 2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
      v[8 * h + 2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = warp_max(amax);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = e4m3_code(__fdiv_rn(v[4 * i], scale)) | (e4m3_code(__fdiv_rn(v[4 * i + 1], scale)) << 8) |
           (e4m3_code(__fdiv_rn(v[4 * i + 2], scale)) << 16) | (e4m3_code(__fdiv_rn(v[4 * i + 3], scale)) << 24);
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
  if (lane == 0) *reinterpret_cast<float*>(dst + 512) = scale;
  if (lane >= 1 && lane <= 3) reinterpret_cast<uint32_t*>(dst + 512)[lane] = 0u;   // bytes [516, 528)
  if (lane < 8) reinterpret_cast<uint4*>(dst + 528)[lane] = __ldg(src + 64 + lane);  // rope
}

// 656-byte FP8 rows with one power-of-two scale per 128 latent dims: lane l holds
// latent values [16 l, 16 l + 16), tile l / 8, whose amax is a 3-step shuffle max.
__global__ void __launch_bounds__(kAppendWarps * 32)
    latent_fp8_tile_kernel(SeqArgs seq, int64_t row_bytes, const uint16_t* kv_new, uint8_t* cache) {
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAppendWarps + warp;
  if (t >= seq.T) return;
  const int64_t row = append_row(seq, t);
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(kv_new + static_cast<int64_t>(t) * 576);
  uint8_t* dst = cache + row * row_bytes;
  float v[16];
  float amax = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 u = __ldg(src + 2 * lane + h);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * h + 2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
      v[8 * h + 2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int e = mx_exponent(amax);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = e4m3_code(ldexpf(v[4 * i], -e)) | (e4m3_code(ldexpf(v[4 * i + 1], -e)) << 8) |
           (e4m3_code(ldexpf(v[4 * i + 2], -e)) << 16) | (e4m3_code(ldexpf(v[4 * i + 3], -e)) << 24);
  reinterpret_cast<uint4*>(dst)[lane] = make_uint4(q[0], q[1], q[2], q[3]);
  if ((lane & 7) == 0) reinterpret_cast<float*>(dst + 512)[lane >> 3] = ldexpf(1.f, e);
  if (lane < 8) reinterpret_cast<uint4*>(dst + 528)[lane] = __ldg(src + 64 + lane);  // rope
}

}  // namespace

cudaError_t launch_index_append_mx(const SeqArgs& seq, int32_t D, bool bf16_in, const void* k_new, uint8_t* k_cache,
                                   uint8_t* k_exp, const LaunchEnv& env, std::string* plan) {
  if (seq.T == 0) {
    *plan += "index_append_mx[empty]";
    return cudaSuccess;
  }
  const dim3 grid((seq.T + kAppendWarps - 1) / kAppendWarps), block(kAppendWarps * 32);
  const cudaError_t e =
      bf16_in ? launch_kernel(index_append_mx_kernel<true>, grid, block, 0, env.stream, true, 1, seq, D, k_new, k_cache,
                              k_exp)
              : launch_kernel(index_append_mx_kernel<false>, grid, block, 0, env.stream, true, 1, seq, D, k_new,
                              k_cache, k_exp);
  *plan += bf16_in ? "index_append_mx<bf16>" : "index_append_mx<f32>";
  return e;
}

cudaError_t launch_index_append(const SeqArgs& seq, int32_t D, bool bf16_in, const void* k_new, uint8_t* k_cache,
                                float* k_scale, const LaunchEnv& env, std::string* plan) {
  if (seq.T == 0) {
    *plan += "index_append[empty]";
    return cudaSuccess;
  }
  const dim3 grid((seq.T + kAppendWarps - 1) / kAppendWarps), block(kAppendWarps * 32);
  const cudaError_t e =
      bf16_in ? launch_kernel(index_append_kernel<true>, grid, block, 0, env.stream, true, 1, seq, D, k_new, k_cache,
                              k_scale)
              : launch_kernel(index_append_kernel<false>, grid, block, 0, env.stream, true, 1, seq, D, k_new, k_cache,
                              k_scale);
  *plan += bf16_in ? "index_append<bf16>" : "index_append<f32>";
  return e;
}

cudaError_t launch_latent_append(const SeqArgs& seq, const MlaArgs& a, const void* kv_new, void* kv_cache,
                                 const LaunchEnv& env, std::string* plan) {
  if (seq.T == 0) {
    *plan += "latent_append[empty]";
    return cudaSuccess;
  }
  const dim3 grid((seq.T + kAppendWarps - 1) / kAppendWarps), block(kAppendWarps * 32);
  uint8_t* cache = static_cast<uint8_t*>(kv_cache);
  if (a.kind == MlaKind::kFP8Tile) {
    *plan += "latent_append<fp8_tile128>";
    return launch_kernel(latent_fp8_tile_kernel, grid, block, 0, env.stream, true, 1, seq, a.row_bytes,
                         static_cast<const uint16_t*>(kv_new), cache);
  }
  if (a.kind == MlaKind::kFP8Row) {
    *plan += "latent_append<fp8_row>";
    return launch_kernel(latent_fp8_kernel, grid, block, 0, env.stream, true, 1, seq, a.row_bytes,
                         static_cast<const uint16_t*>(kv_new), cache);
  }
  const int64_t row_in = static_cast<int64_t>(a.d_latent + a.d_rope) * (a.kind == MlaKind::kF32 ? 4 : 2);
  *plan += a.kind == MlaKind::kF32 ? "latent_append<f32>" : "latent_append<bf16>";
  return launch_kernel(latent_copy_kernel, grid, block, 0, env.stream, true, 1, seq, row_in, a.row_bytes, kv_new,
                       cache);
}

}  // namespace dsa
