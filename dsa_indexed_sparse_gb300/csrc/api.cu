// C-ABI facade of libdsa: host-side validation, kernel choice, workspace layout
// and the chained decode step.  Every entry point returns a dsa_status_t and
// never lets a C++ exception escape.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "dsa.h"
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace {

thread_local std::string g_last_error;
thread_local std::string g_last_plan;

dsa_status_t fail(dsa_status_t s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

dsa_status_t cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return DSA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device SM count, cached.
int num_sms_for(int device) {
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (device < 0 || device >= 64) return 148;
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
      n = 148;
    cache[device] = n;
  }
  return cache[device];
}

dsa_status_t make_env(dsa_stream_t stream, dsa::LaunchEnv* env) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  env->stream = static_cast<cudaStream_t>(stream);
  env->device = dev;
  env->num_sms = num_sms_for(dev);
  return DSA_OK;
}

dsa_status_t check_seq(const dsa_seq_desc_t* s, dsa::SeqArgs* out) {
  if (!s) return fail(DSA_ERR_INVALID_ARG, "seq descriptor is NULL");
  if (s->T < 0 || s->B < 1) return fail(DSA_ERR_INVALID_ARG, "need T >= 0 and B >= 1");
  if (s->max_ctx < 1) return fail(DSA_ERR_INVALID_ARG, "max_ctx must be >= 1");
  if (s->page_size < 1) return fail(DSA_ERR_INVALID_ARG, "page_size must be >= 1");
  if (s->q_per_seq < 0) return fail(DSA_ERR_INVALID_ARG, "q_per_seq must be >= 0");
  if (s->q_per_seq > 0 && static_cast<int64_t>(s->B) * s->q_per_seq != s->T)
    return fail(DSA_ERR_INVALID_ARG, "q_per_seq > 0 requires T == B * q_per_seq");
  const int64_t pages_needed = (static_cast<int64_t>(s->max_ctx) + s->page_size - 1) / s->page_size;
  if (s->bt_stride < pages_needed)
    return fail(DSA_ERR_INVALID_ARG, "bt_stride < ceil(max_ctx / page_size)");
  if (s->cache_rows < s->page_size || s->cache_rows % s->page_size != 0)
    return fail(DSA_ERR_INVALID_ARG, "cache_rows must be a positive multiple of page_size");
  if (s->cache_rows > 0x7FFFFFFFll) return fail(DSA_ERR_INVALID_ARG, "cache_rows >= 2^31");
  if (s->T > 0 && (!s->q_seq || !s->q_pos || !s->block_table))
    return fail(DSA_ERR_INVALID_ARG, "q_seq, q_pos and block_table must be non-NULL");
  *out = dsa::SeqArgs{s->B, s->T, s->max_ctx, s->q_per_seq, s->q_seq, s->q_pos, s->block_table,
                      s->bt_stride, s->page_size, s->cache_rows, s->cache_rows / s->page_size};
  return DSA_OK;
}

dsa_status_t check_indexer(const dsa_seq_desc_t* s, const dsa_indexer_desc_t* x, const float* scores,
                           int64_t ld, dsa::IndexerArgs* out) {
  if (!x) return fail(DSA_ERR_INVALID_ARG, "indexer descriptor is NULL");
  if (x->H_I < 1 || x->D_I < 1) return fail(DSA_ERR_INVALID_ARG, "H_I and D_I must be >= 1");
  if (x->dtype != DSA_E4M3 && x->dtype != DSA_F32 && x->dtype != DSA_MXFP8_E4M3)
    return fail(DSA_ERR_UNSUPPORTED, "indexer dtype must be DSA_E4M3, DSA_MXFP8_E4M3 or DSA_F32");
  const bool mx = x->dtype == DSA_MXFP8_E4M3;
  if (mx && x->D_I % 32 != 0) return fail(DSA_ERR_UNSUPPORTED, "MXFP8 index keys need D_I a multiple of 32");
  if (s->T > 0 && (!x->q || !x->w || !x->k_cache))
    return fail(DSA_ERR_INVALID_ARG, "indexer q, w and k_cache must be non-NULL");
  if (s->T > 0 && mx && (!x->q_scale || !x->k_scale))
    return fail(DSA_ERR_INVALID_ARG, "MXFP8 index keys need q_scale and k_scale");
  if (!aligned16(x->q) || !aligned16(x->k_cache) || !aligned16(x->w) || !aligned16(x->q_scale) ||
      !aligned16(x->k_scale))
    return fail(DSA_ERR_INVALID_ARG, "indexer pointers must be 16-byte aligned");
  if (ld < s->max_ctx || ld % 4 != 0) return fail(DSA_ERR_INVALID_ARG, "ld must be >= max_ctx and a multiple of 4");
  if (s->T > 0 && (!scores || !aligned16(scores)))
    return fail(DSA_ERR_INVALID_ARG, "scores must be non-NULL and 16-byte aligned");
  *out = dsa::IndexerArgs{x->H_I, x->D_I, x->dtype != DSA_F32, mx, x->q, x->q_scale, x->w,
                          x->k_cache, x->k_scale, const_cast<float*>(scores), ld};
  return DSA_OK;
}

// Shape/format checks only (no pointers): fills *a with null data pointers.
dsa_status_t check_mla_shape(const dsa_mla_desc_t* m, int32_t K, dsa::MlaArgs* a) {
  if (!m) return fail(DSA_ERR_INVALID_ARG, "mla descriptor is NULL");
  if (m->H < 1 || m->d_latent < 1 || m->d_rope < 0)
    return fail(DSA_ERR_INVALID_ARG, "need H >= 1, d_latent >= 1, d_rope >= 0");
  if (K < 1 || K > 16384) return fail(DSA_ERR_UNSUPPORTED, "K must be in [1, 16384]");
  const int64_t dqk = static_cast<int64_t>(m->d_latent) + m->d_rope;
  dsa::MlaKind kind;
  int64_t min_row;
  switch (m->dtype) {
    case DSA_F32: kind = dsa::MlaKind::kF32; min_row = 4 * dqk; break;
    case DSA_BF16: kind = dsa::MlaKind::kBF16; min_row = 2 * dqk; break;
    case DSA_E4M3:
      if (m->d_latent != 512 || m->d_rope != 64)
        return fail(DSA_ERR_UNSUPPORTED, "FP8 latent rows are defined for 512 + 64 dims only");
      kind = dsa::MlaKind::kFP8Row;
      min_row = 656;
      break;
    case DSA_E4M3_T128:
      if (m->d_latent != 512 || m->d_rope != 64)
        return fail(DSA_ERR_UNSUPPORTED, "FP8 latent rows are defined for 512 + 64 dims only");
      kind = dsa::MlaKind::kFP8Tile;
      min_row = 656;
      break;
    default: return fail(DSA_ERR_UNSUPPORTED, "unknown MLA cache dtype");
  }
  if (m->row_bytes < min_row) return fail(DSA_ERR_INVALID_ARG, "row_bytes smaller than one row");
  if (m->row_bytes % (kind == dsa::MlaKind::kBF16 ? 2 : 4) != 0)
    return fail(DSA_ERR_INVALID_ARG, "row_bytes not a multiple of the element size");
  *a = dsa::MlaArgs{m->H, m->d_latent, m->d_rope, kind, m->q, m->kv_cache, m->row_bytes,
                    m->softmax_scale, nullptr, K, nullptr, nullptr};
  return DSA_OK;
}

dsa_status_t check_mla(const dsa_seq_desc_t* s, const dsa_mla_desc_t* m, const int32_t* idx, int32_t K,
                       void* out, float* lse, dsa::MlaArgs* a) {
  dsa_status_t st = check_mla_shape(m, K, a);
  if (st != DSA_OK) return st;
  if (s->T > 0 && (!m->q || !m->kv_cache || !idx || !out))
    return fail(DSA_ERR_INVALID_ARG, "q, kv_cache, idx and out must be non-NULL");
  if (!aligned16(m->q) || !aligned16(m->kv_cache) || !aligned16(idx) || !aligned16(out) || !aligned16(lse))
    return fail(DSA_ERR_INVALID_ARG, "MLA pointers must be 16-byte aligned");
  a->idx = idx;
  a->out = out;
  a->lse = lse;
  return DSA_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

namespace dsa {

void set_last_error(const std::string& msg) { g_last_error = msg; }

cudaError_t ensure_smem_limit(const void* kernel, int bytes, int device) {
  struct Entry {
    const void* kernel;
    int device;
    cudaError_t result;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : done)
    if (e.kernel == kernel && e.device == device) return e.result;
  const cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  done.push_back(Entry{kernel, device, r});
  return r;
}

bool cluster_fits(const void* kernel, int device, int cl, int threads, size_t smem) {
  struct Entry {
    const void* kernel;
    int device, cl, threads;
    size_t smem;
    bool fits;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& e : done)
    if (e.kernel == kernel && e.device == device && e.cl == cl && e.threads == threads && e.smem == smem)
      return e.fits;
  if (cl > 8) static_cast<void>(cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cl));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cl);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  const bool fits = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n >= 1;
  cudaGetLastError();
  done.push_back(Entry{kernel, device, cl, threads, smem, fits});
  return fits;
}

namespace {
std::atomic<uint32_t> g_dbg_withhold{0};
std::atomic<uint64_t> g_dbg_wait_limit_ns{kWaitLimitNs};
}  // namespace

void debug_wait_state(uint64_t* wait_limit_ns, uint32_t* withhold) {
  *wait_limit_ns = g_dbg_wait_limit_ns.load(std::memory_order_relaxed);
  *withhold = g_dbg_withhold.load(std::memory_order_relaxed);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
bool encode_tmap_2d_u8(void* tmap_out, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       std::string* why) {
  return encode_tmap_2d(tmap_out, base, 1, inner, rows, row_stride_bytes, box_inner, box_rows, why);
}

bool encode_tmap_2d(void* tmap_out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, std::string* why) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  if (!fn) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), dt, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    *why = buf;
    return false;
  }
  return true;
}

}  // namespace dsa

extern "C" {

int dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT";
    case DSA_ERR_DEVICE_CHECK: return "DSA_ERR_DEVICE_CHECK";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error(void) { return g_last_error.c_str(); }
const char* dsa_last_plan(void) { return g_last_plan.c_str(); }

dsa_status_t dsa_indexer_scores(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx, float* scores,
                                int64_t ld, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa::IndexerArgs a;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if ((st = check_indexer(seq, idx, scores, ld, &a)) != DSA_OK) return st;
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan, why;
    bool unsupported = false;
    cudaError_t e = dsa::launch_indexer(s, a, env, &plan, &unsupported, &why);
    if (unsupported) return fail(DSA_ERR_UNSUPPORTED, why);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

dsa_status_t dsa_topk(const dsa_seq_desc_t* seq, const float* scores, int64_t ld, int32_t K, int32_t* idx,
                      dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if (K < 1) return fail(DSA_ERR_INVALID_ARG, "K must be >= 1");
    if (ld < s.max_ctx || ld % 4 != 0) return fail(DSA_ERR_INVALID_ARG, "ld must be >= max_ctx and a multiple of 4");
    if (s.T > 0 && (!scores || !idx)) return fail(DSA_ERR_INVALID_ARG, "scores and idx must be non-NULL");
    if (!aligned16(scores)) return fail(DSA_ERR_INVALID_ARG, "scores must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan;
    cudaError_t e = dsa::launch_topk(s, scores, ld, K, idx, env, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "topk launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

size_t dsa_sparse_mla_attn_workspace_size(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, int32_t K) {
  try {
    dsa::SeqArgs s;
    dsa::MlaArgs a;
    if (check_seq(seq, &s) != DSA_OK) return 0;
    if (check_mla_shape(mla, K, &a) != DSA_OK) return 0;
    dsa::LaunchEnv env;
    if (make_env(nullptr, &env) != DSA_OK) return 0;
    return dsa::attn_workspace_bytes(s, a, env.num_sms);
  } catch (...) {
    return 0;
  }
}

dsa_status_t dsa_sparse_mla_attn(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, const int32_t* idx,
                                 int32_t K, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa::MlaArgs a;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if ((st = check_mla(seq, mla, idx, K, out, lse, &a)) != DSA_OK) return st;
    if (workspace && !aligned16(workspace)) return fail(DSA_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan, why;
    bool unsupported = false;
    cudaError_t e = dsa::launch_attn(s, a, workspace, workspace ? workspace_bytes : 0, env, &plan,
                                     &unsupported, &why);
    if (unsupported) return fail(DSA_ERR_UNSUPPORTED, why);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

// Workspace of the chained step: [scores T x ld fp32][idx T x K int32][attention partials].
static size_t decode_ws_layout(const dsa::SeqArgs& s, const dsa::MlaArgs& a, int num_sms, int64_t* ld,
                               size_t* off_idx, size_t* off_attn) {
  *ld = (static_cast<int64_t>(s.max_ctx) + 3) / 4 * 4;
  const size_t scores = align256(static_cast<size_t>(s.T) * *ld * sizeof(float));
  const size_t idx = align256(static_cast<size_t>(s.T) * a.K * sizeof(int32_t));
  *off_idx = scores;
  *off_attn = scores + idx;
  return scores + idx + dsa::attn_workspace_bytes(s, a, num_sms);
}

}  // extern "C"

namespace dsa {
dsa_status_t decode_workspace_need(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, int32_t K, size_t* need) {
  *need = 0;
  try {
    dsa::SeqArgs s;
    dsa::MlaArgs a;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if ((st = check_mla_shape(mla, K, &a)) != DSA_OK) return st;
    dsa::LaunchEnv env;
    if ((st = make_env(nullptr, &env)) != DSA_OK) return st;
    int64_t ld;
    size_t oi, oa;
    *need = decode_ws_layout(s, a, env.num_sms, &ld, &oi, &oa);
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}
}  // namespace dsa

extern "C" {

size_t dsa_decode_workspace_size(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx,
                                 const dsa_mla_desc_t* mla, int32_t K) {
  (void)idx;
  size_t need = 0;
  return dsa::decode_workspace_need(seq, mla, K, &need) == DSA_OK ? need : 0;
}

dsa_status_t dsa_decode_step(const dsa_seq_desc_t* seq, const dsa_indexer_desc_t* idx, const dsa_mla_desc_t* mla,
                             int32_t K, void* out, float* lse, int32_t* idx_out, void* workspace,
                             size_t workspace_bytes, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if (!workspace || !aligned16(workspace)) return fail(DSA_ERR_WORKSPACE, "workspace must be non-NULL and 16-byte aligned");
    if (idx_out && !aligned16(idx_out)) return fail(DSA_ERR_INVALID_ARG, "idx_out must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    dsa::MlaArgs a;
    if ((st = check_mla_shape(mla, K, &a)) != DSA_OK) return st;
    int64_t ld;
    size_t off_idx, off_attn;
    const size_t need = decode_ws_layout(s, a, env.num_sms, &ld, &off_idx, &off_attn);
    if (workspace_bytes < need) {
      char buf[128];
      snprintf(buf, sizeof(buf), "workspace too small: %zu < %zu bytes", workspace_bytes, need);
      return fail(DSA_ERR_WORKSPACE, buf);
    }
    char* ws = static_cast<char*>(workspace);
    float* scores = reinterpret_cast<float*>(ws);
    int32_t* sel = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + off_idx);
    dsa::IndexerArgs ia;
    if ((st = check_indexer(seq, idx, scores, ld, &ia)) != DSA_OK) return st;
    if ((st = check_mla(seq, mla, sel, K, out, lse, &a)) != DSA_OK) return st;

    std::string plan, why;
    bool unsupported = false;
    // fused plan (scores stay in shared memory) when the batch and contexts allow
    cudaError_t e = dsa::launch_decode_fused(s, ia, K, sel, env, &plan, &unsupported, &why);
    if (e != cudaSuccess) return cuda_fail(e, "fused indexer + top-k launch");
    if (unsupported) {
      plan.clear();
      e = dsa::launch_indexer(s, ia, env, &plan, &unsupported, &why);
      if (unsupported) return fail(DSA_ERR_UNSUPPORTED, why);
      if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
      plan += " -> ";
      e = dsa::launch_topk(s, scores, ld, K, sel, env, &plan);
      if (e != cudaSuccess) return cuda_fail(e, "topk launch");
    }
    plan += " -> ";
    e = dsa::launch_attn(s, a, ws + off_attn, workspace_bytes - off_attn, env, &plan, &unsupported, &why);
    if (unsupported) return fail(DSA_ERR_UNSUPPORTED, why);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

dsa_status_t dsa_index_cache_append(const dsa_seq_desc_t* seq, int32_t D_I, dsa_dtype_t src_dtype,
                                    const void* k_new, uint8_t* k_cache, float* k_scale, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if (D_I < 4 || D_I > 1024 || D_I % 4 != 0)
      return fail(DSA_ERR_UNSUPPORTED, "index-key append needs D_I in [4, 1024], a multiple of 4");
    if (src_dtype != DSA_F32 && src_dtype != DSA_BF16)
      return fail(DSA_ERR_UNSUPPORTED, "new index keys must be DSA_F32 or DSA_BF16");
    if (s.T > 0 && (!k_new || !k_cache || !k_scale))
      return fail(DSA_ERR_INVALID_ARG, "k_new, k_cache and k_scale must be non-NULL");
    if (!aligned16(k_new) || !aligned16(k_cache) || !aligned16(k_scale))
      return fail(DSA_ERR_INVALID_ARG, "k_new, k_cache and k_scale must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan;
    cudaError_t e = dsa::launch_index_append(s, D_I, src_dtype == DSA_BF16, k_new, k_cache, k_scale, env, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "index-key append launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

dsa_status_t dsa_index_cache_append_mx(const dsa_seq_desc_t* seq, int32_t D_I, dsa_dtype_t src_dtype,
                                       const void* k_new, uint8_t* k_cache, uint8_t* k_exp, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if (D_I < 32 || D_I > 1024 || D_I % 32 != 0)
      return fail(DSA_ERR_UNSUPPORTED, "MXFP8 index-key append needs D_I in [32, 1024], a multiple of 32");
    if (src_dtype != DSA_F32 && src_dtype != DSA_BF16)
      return fail(DSA_ERR_UNSUPPORTED, "new index keys must be DSA_F32 or DSA_BF16");
    if (s.T > 0 && (!k_new || !k_cache || !k_exp))
      return fail(DSA_ERR_INVALID_ARG, "k_new, k_cache and k_exp must be non-NULL");
    if (!aligned16(k_new) || !aligned16(k_cache) || !aligned16(k_exp))
      return fail(DSA_ERR_INVALID_ARG, "k_new, k_cache and k_exp must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan;
    cudaError_t e = dsa::launch_index_append_mx(s, D_I, src_dtype == DSA_BF16, k_new, k_cache, k_exp, env, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "index-key append launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

dsa_status_t dsa_latent_cache_append(const dsa_seq_desc_t* seq, const dsa_mla_desc_t* mla, const void* kv_new,
                                     void* kv_cache, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa::MlaArgs a;
    dsa_status_t st = check_seq(seq, &s);
    if (st != DSA_OK) return st;
    if ((st = check_mla_shape(mla, 1, &a)) != DSA_OK) return st;
    if (a.kind != dsa::MlaKind::kFP8Row && a.kind != dsa::MlaKind::kFP8Tile) {
      const int64_t row_in = static_cast<int64_t>(a.d_latent + a.d_rope) * (a.kind == dsa::MlaKind::kF32 ? 4 : 2);
      if (row_in % 16 != 0 || a.row_bytes % 16 != 0)
        return fail(DSA_ERR_UNSUPPORTED, "latent append copies 16-byte vectors: row and row_bytes must be multiples of 16");
    } else if (a.row_bytes % 16 != 0) {
      return fail(DSA_ERR_INVALID_ARG, "row_bytes must be a multiple of 16");
    }
    if (s.T > 0 && (!kv_new || !kv_cache)) return fail(DSA_ERR_INVALID_ARG, "kv_new and kv_cache must be non-NULL");
    if (!aligned16(kv_new) || !aligned16(kv_cache))
      return fail(DSA_ERR_INVALID_ARG, "kv_new and kv_cache must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    std::string plan;
    cudaError_t e = dsa::launch_latent_append(s, a, kv_new, kv_cache, env, &plan);
    if (e != cudaSuccess) return cuda_fail(e, "latent append launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

namespace {
dsa_status_t check_prolog(const dsa_seq_desc_t* seq, const dsa_prolog_desc_t* pd, dsa::SeqArgs* s) {
  dsa_status_t st = check_seq(seq, s);
  if (st != DSA_OK) return st;
  if (!pd) return fail(DSA_ERR_INVALID_ARG, "prolog descriptor is NULL");
  if (pd->D_I != 128) return fail(DSA_ERR_UNSUPPORTED, "the prolog kernels need D_I == 128");
  if (pd->H_I < 1 || pd->H_I > 128) return fail(DSA_ERR_UNSUPPORTED, "the prolog kernels need 1 <= H_I <= 128");
  if (pd->d_model < 64 || pd->d_model % 64 != 0 || pd->d_q < 64 || pd->d_q % 64 != 0)
    return fail(DSA_ERR_UNSUPPORTED, "d_model and d_q must be positive multiples of 64");
  return DSA_OK;
}
}  // namespace

size_t dsa_indexer_prolog_workspace_size(const dsa_seq_desc_t* seq, const dsa_prolog_desc_t* pd) {
  try {
    dsa::SeqArgs s;
    if (check_prolog(seq, pd, &s) != DSA_OK) return 0;
    dsa::LaunchEnv env;
    if (make_env(nullptr, &env) != DSA_OK) return 0;
    return dsa::prolog_workspace_bytes(s.T, pd->H_I, pd->d_model, pd->d_q, env.num_sms);
  } catch (...) {
    return 0;
  }
}

dsa_status_t dsa_indexer_prolog(const dsa_seq_desc_t* seq, const dsa_prolog_desc_t* pd, uint8_t* q_codes,
                                float* q_scale, float* w, uint8_t* k_cache, float* k_scale, void* workspace,
                                size_t workspace_bytes, dsa_stream_t stream) {
  try {
    dsa::SeqArgs s;
    dsa_status_t st = check_prolog(seq, pd, &s);
    if (st != DSA_OK) return st;
    if (s.T > 0 && (!pd->x || !pd->x_q || !pd->w_q || !pd->w_k || !pd->w_w || !pd->gamma || !pd->beta ||
                    !q_codes || !q_scale || !w || !k_cache || !k_scale))
      return fail(DSA_ERR_INVALID_ARG, "prolog inputs and outputs must be non-NULL");
    if (!aligned16(pd->x) || !aligned16(pd->x_q) || !aligned16(pd->w_q) || !aligned16(pd->w_k) ||
        !aligned16(pd->w_w) || !aligned16(q_codes) || !aligned16(q_scale) || !aligned16(w) || !aligned16(k_cache) ||
        !aligned16(k_scale))
      return fail(DSA_ERR_INVALID_ARG, "prolog pointers must be 16-byte aligned");
    dsa::LaunchEnv env;
    if ((st = make_env(stream, &env)) != DSA_OK) return st;
    const size_t need = dsa::prolog_workspace_bytes(s.T, pd->H_I, pd->d_model, pd->d_q, env.num_sms);
    if (s.T > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need)) {
      char buf[128];
      snprintf(buf, sizeof(buf), "prolog workspace: need %zu bytes, 16-byte aligned", need);
      return fail(DSA_ERR_WORKSPACE, buf);
    }
    const dsa::PrologArgs a{pd->d_model, pd->d_q, pd->H_I, pd->x, pd->x_q, pd->w_q, pd->w_k, pd->w_w, pd->gamma,
                            pd->beta, q_codes, q_scale, w, k_cache, k_scale};
    std::string plan, why;
    bool unsupported = false;
    const cudaError_t e = dsa::launch_prolog(s, a, workspace, env, &plan, &unsupported, &why);
    if (unsupported) return fail(DSA_ERR_UNSUPPORTED, why);
    if (e != cudaSuccess) return cuda_fail(e, "prolog launch");
    g_last_plan = plan;
    return DSA_OK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

dsa_status_t dsa_debug_withhold_arrival(int32_t enable, uint64_t wait_limit_ns) {
  if (enable && (wait_limit_ns < 1000ull || wait_limit_ns > dsa::kWaitLimitNs))
    return fail(DSA_ERR_INVALID_ARG, "wait_limit_ns must be in [1 us, 1 s]");
  dsa::g_dbg_wait_limit_ns.store(enable ? wait_limit_ns : dsa::kWaitLimitNs, std::memory_order_relaxed);
  dsa::g_dbg_withhold.store(enable ? 1u : 0u, std::memory_order_relaxed);
  return DSA_OK;
}

dsa_status_t dsa_check_status(dsa_stream_t stream) {
  try {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    const uint32_t f = dsa_status_read_clear_indexer() | dsa_status_read_clear_topk() |
                       dsa_status_read_clear_attn() | dsa_status_read_clear_cache() |
                       dsa_status_read_clear_prolog();
    if (f == 0) return DSA_OK;
    if (f == 0xFFFFFFFFu) return fail(DSA_ERR_CUDA, "could not read the device status word");
    std::string msg = "device flags:";
    if (f & dsa::kDevTimeout) msg += " timeout";
    if (f & dsa::kDevBadIndex) msg += " bad_index";
    if (f & dsa::kDevBadPos) msg += " bad_q_pos";
    if (f & dsa::kDevBadGroup) msg += " bad_q_per_seq";
    if (f & dsa::kDevConfig) msg += " launch_config";
    g_last_error = msg;
    return (f & dsa::kDevTimeout) ? DSA_ERR_TIMEOUT : DSA_ERR_DEVICE_CHECK;
  } catch (...) {
    return fail(DSA_ERR_CUDA, "unexpected host exception");
  }
}

}  // extern "C"
