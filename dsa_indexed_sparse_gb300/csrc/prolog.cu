// The indexer prolog: the lightning indexer's query, head weights and new key made
// from the new tokens' hidden states.
//
// "Large Language Model Inference Acceleration in Practice", section 3.2 "Indexer
// Prolog": the input preparation before the indexer is a query projection, a key
// normalisation with the key-cache update, a query quantisation and a head-weight
// projection; the pages run them on three streams so that they overlap.  Here
//   q[t]  = W_q x_q[t]                      (H_I heads of D_I = 128 values)
//   w[t]  = W_w x[t]                        (H_I head weights)
//   k[t]  = LayerNorm(W_k x[t]) * gamma + beta   (population variance, eps 1e-6)
// with bf16 inputs and weights and fp32 accumulation; each query head and the
// key are quantised to E4M3 with one fp32 scale (amax / 448, round to nearest
// even, saturated -- the cache formats' rule) and the key is written to the
// cache row of its position.  On one GPU the pages' three streams become one
// grid: every projection tile of the three weights is a CTA of the same launch.
//
// Two kernels:
//  * prolog_proj_kernel -- tcgen05 bf16 GEMM, swap-AB: a CTA multiplies 128 rows
//    of one weight (output features; M) by up to 256 tokens (N), over a range of
//    64-wide K atoms (split-K when the batch is small: each K range writes its
//    own fp32 slice of the workspace, no atomics and no zeroing); weights and
//    tokens arrive by 2-D TMA (128-byte swizzle), the accumulator lives in TMEM.
//  * prolog_epilogue_kernel -- one warp per (token, query head): the slices'
//    sum, the per-head query quantisation; one more warp per token for the key's
//    layer normalisation, quantisation and cache write, and the head weights.
#include <algorithm>
#include <cmath>
#include <cstdio>

#include "dsa_device.cuh"
#include "dsa_internal.h"

DSA_DEFINE_STATUS_WORD(prolog)

namespace dsa {
namespace {

constexpr int kPM = 128;           // output features per CTA (UMMA M)
constexpr int kPAtom = 64;         // bf16 elements per K atom (one 128-byte swizzle row)
constexpr int kPMaxN = 256;        // tokens per CTA at most (UMMA N)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;     // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kPABytes = kPM * kPAtom * 2;             // 16 KB
constexpr int kPNumBars = 2 * kPStages + 2;            // full, empty, accfull, drain
// Shared memory of a CTA for n_tok tokens: kPStages x (weight tile + token tile),
// barriers, misc words, re-alignment slack.  Sized by the token tile so that two
// CTAs share an SM at small batches (two independent issue chains per SM).
__host__ __device__ constexpr int prolog_stage_bytes(int n_tok) { return kPABytes + n_tok * kPAtom * 2; }
__host__ __device__ constexpr int prolog_smem_bytes(int n_tok) {
  return kPStages * prolog_stage_bytes(n_tok) + kPNumBars * 8 + 64 + 1024;
}

struct ProjJob {
  int32_t n_feat;      // output features of this weight
  int32_t k_atoms;     // reduction length / 64
  int32_t split;       // K ranges per (feature tile, token tile)
  int32_t f_tiles;     // ceil(n_feat / 128)
  int32_t first_cta;   // first CTA index of this job
  float* y;            // fp32 [split][T, ld] (+ column offset)
  int32_t ld;
  int64_t slice;       // elements between two K ranges' slices
};

struct ProjParams {
  int32_t T;
  int32_t n_tok;       // tokens per CTA (multiple of 16, <= 256)
  uint32_t tmem_cols;  // power of two >= n_tok, >= 32
  int32_t t_tiles;
  ProjJob job[3];      // 0: query (W_q, x_q), 1: key (W_k, x), 2: head weights (W_w, x)
  uint64_t wait_limit_ns;
};

__global__ void __launch_bounds__(kPThreads, 2)
    prolog_proj_kernel(const __grid_constant__ CUtensorMap wq_map, const __grid_constant__ CUtensorMap wk_map,
                       const __grid_constant__ CUtensorMap ww_map, const __grid_constant__ CUtensorMap xq_map,
                       const __grid_constant__ CUtensorMap x_map, ProjParams p) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  const int stage_bytes = prolog_stage_bytes(p.n_tok);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kPStages * stage_bytes);
  uint64_t* empty = full + kPStages;
  uint64_t* accfull = empty + kPStages;
  uint64_t* drain = accfull + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t wlim = p.wait_limit_ns;

  // ---- which tile: job, feature tile, token tile, K range ----------------
  // grid order: key tiles, head-weight tiles, query tiles (the longer reductions first)
  const int cta = static_cast<int>(blockIdx.x);
  const int jb = cta >= p.job[0].first_cta ? 0 : (cta >= p.job[2].first_cta ? 2 : 1);
  const ProjJob& J = p.job[jb];
  int r = cta - J.first_cta;
  const int sp = r % J.split;
  r /= J.split;
  const int tt = r % p.t_tiles;
  const int ft = r / p.t_tiles;
  const int a0 = static_cast<int>(static_cast<int64_t>(sp) * J.k_atoms / J.split);
  const int a1 = static_cast<int>(static_cast<int64_t>(sp + 1) * J.k_atoms / J.split);
  const int n_atoms = a1 - a0;
  const CUtensorMap* amap = jb == 0 ? &wq_map : (jb == 1 ? &wk_map : &ww_map);
  const CUtensorMap* bmap = jb == 0 ? &xq_map : &x_map;
  const int f0 = ft * kPM, t0 = tt * p.n_tok;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(accfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(amap);
    tma_prefetch_desc(bmap);
  }
  if (warp == 1) {
    tmem_alloc(misc, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  grid_dep_wait();   // the inputs may come from the kernel before

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    const uint32_t bytes = kPABytes + static_cast<uint32_t>(p.n_tok) * kPAtom * 2;
    int issued = 0;
    for (int i = 0; i < n_atoms; ++i) {
      const int st = i % kPStages;
      if (i >= kPStages) {
        const bool ok = mbar_wait(&empty[st], ((i / kPStages) - 1) & 1, &g_status_prolog, abort_flag, wlim);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) {
        uint8_t* a = sm + st * stage_bytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        tma_load_2d(a, amap, &full[st], (a0 + i) * kPAtom, f0);
        tma_load_2d(a + kPABytes, bmap, &full[st], (a0 + i) * kPAtom, t0);
      }
      __syncwarp();
      ++issued;
    }
    for (int m = 0; m < min(issued, kPStages); ++m) {
      const int k = issued - 1 - m;
      mbar_drain(&full[k % kPStages], (k / kPStages) & 1, &g_status_prolog, wlim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, false, false, kPM, static_cast<uint32_t>(p.n_tok));
    for (int i = 0; i < n_atoms; ++i) {
      const int st = i % kPStages;
      const bool ok = mbar_wait(&full[st], (i / kPStages) & 1, &g_status_prolog, abort_flag, wlim);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint64_t da = make_sdesc(smem_u32(sm + st * stage_bytes), 16, 1024, kLayoutSw128);
      const uint64_t db = make_sdesc(smem_u32(sm + st * stage_bytes + kPABytes), 16, 1024, kLayoutSw128);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < kPAtom / 16; ++k)   // 16 bf16 = 32 bytes per step
          umma_f16(tmem, da + static_cast<uint64_t>(2 * k), db + static_cast<uint64_t>(2 * k), idesc,
                   (i > 0 || k > 0) ? 1u : 0u);
        umma_commit(&empty[st]);
        if (i == n_atoms - 1) umma_commit(accfull);
      }
      __syncwarp();
    }
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    mbar_drain(drain, 0, &g_status_prolog, wlim);
  } else {
    // ------------------------------------------------ epilogue: TMEM -> y
    // thread = one output feature (its TMEM lane); 32 tokens per TMEM load
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int f = f0 + row;
    bool ok = n_atoms > 0 && mbar_wait(accfull, 0, &g_status_prolog, abort_flag, wlim);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      for (int c0 = 0; c0 < p.n_tok; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + c0, v);
        tmem_ld_wait();
        if (f < J.n_feat) {
          float* y = J.y + sp * J.slice + f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int t = t0 + c0 + j;
            if (t < p.T) y[static_cast<int64_t>(t) * J.ld] = __uint_as_float(v[j]);
          }
        }
      }
    }
  }
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// E4M3 code of a float (round to nearest even, magnitudes beyond 448 saturated).
__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

struct EpiParams {
  SeqArgs seq;
  int32_t H_I;
  const float* yq;     // [split_q][T, H_I * 128]
  int32_t split_q;
  const float* ykw;    // [split_kw][T, 256]: key [0, 128), head weights [128, 128 + H_I)
  int32_t split_kw;
  const float* gamma;
  const float* beta;
  uint8_t* q_codes;    // [T, H_I, 128]
  float* q_scale;      // [T, H_I]
  float* w;            // [T, H_I]
  uint8_t* k_cache;    // [cache_rows, 128]
  float* k_scale;      // [cache_rows]
};

constexpr int kEpiHeads = 16;   // query heads per CTA (one warp each)

// Sum of the K-range slices of one 128-vector: lane l holds values l, l+32,
// l+64, l+96 (a warp's byte stores of one vector are then contiguous).
__device__ __forceinline__ void load_vec128(const float* y, int64_t slice, int split, int lane, float (&v)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = y[lane + 32 * i];
  for (int sp = 1; sp < split; ++sp) {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] += y[sp * slice + lane + 32 * i];
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Grid (T, ceil(H_I / 16) + 1), 16 warps: block row y < last quantises query
// heads 16 y .. 16 y + 15 of token blockIdx.x (a warp each); the last row's warp
// 0 normalises, quantises and stores the token's key, its other warps copy the
// head weights.
__global__ void __launch_bounds__(32 * kEpiHeads) prolog_epilogue_kernel(EpiParams p) {
  grid_dep_wait();
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int HD = p.H_I * 128;
  if (static_cast<int>(blockIdx.y) < static_cast<int>(gridDim.y) - 1) {
    const int h = blockIdx.y * kEpiHeads + warp;
    if (h >= p.H_I) return;
    float v[4];
    load_vec128(p.yq + static_cast<int64_t>(t) * HD + h * 128, static_cast<int64_t>(p.seq.T) * HD, p.split_q,
                lane, v);
    const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    uint8_t* dst = p.q_codes + (static_cast<int64_t>(t) * p.H_I + h) * 128;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = to_e4m3(v[i] / scale);
    if (lane == 0) p.q_scale[static_cast<int64_t>(t) * p.H_I + h] = scale;
    return;
  }
  const int64_t kw_slice = static_cast<int64_t>(p.seq.T) * 256;
  const float* kr = p.ykw + static_cast<int64_t>(t) * 256;
  if (warp > 0) {   // head weights
    for (int h = threadIdx.x - 32; h < p.H_I; h += blockDim.x - 32) {
      float s = kr[128 + h];
      for (int sp = 1; sp < p.split_kw; ++sp) s += kr[sp * kw_slice + 128 + h];
      p.w[static_cast<int64_t>(t) * p.H_I + h] = s;
    }
    return;
  }
  // the key: layer normalisation, quantisation, cache row of its position
  float v[4];
  load_vec128(kr, kw_slice, p.split_kw, lane, v);
  const float mean = warp_sum(v[0] + v[1] + v[2] + v[3]) / 128.f;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss += (v[i] - mean) * (v[i] - mean);
  const float inv = 1.f / sqrtf(warp_sum(ss) / 128.f + 1e-6f);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int d = lane + 32 * i;
    v[i] = (v[i] - mean) * inv * __ldg(p.gamma + d) + __ldg(p.beta + d);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  const int qp = __ldg(p.seq.q_pos + t), b = __ldg(p.seq.q_seq + t);
  if (qp < 0 || qp >= p.seq.max_ctx || b < 0 || b >= p.seq.B) {
    if (lane == 0) atomicOr(&g_status_prolog, kDevBadPos);
    return;
  }
  const int64_t row = phys_row(p.seq.block_table + static_cast<int64_t>(b) * p.seq.bt_stride, qp, p.seq.page_size,
                               p.seq.n_pages, &g_status_prolog);
  if (row < 0) return;
  uint8_t* dst = p.k_cache + row * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = to_e4m3(v[i] / scale);
  if (lane == 0) p.k_scale[row] = scale;
}

int split_for(int tiles, int atoms, int slots) {
  // enough CTAs to fill the resident slots, at least 4 K atoms (256 values) each
  int s = 1;
  while (s * 2 <= atoms / 4 && static_cast<int64_t>(tiles) * s * 2 <= slots) s *= 2;
  return s;
}

}  // namespace

namespace {
struct PrologPlan {
  int n_tok, t_tiles, split_q, split_kw;
  size_t q_bytes, kw_bytes;
};
PrologPlan prolog_plan(int T, int H_I, int d_model, int d_q, int num_sms) {
  PrologPlan pp;
  // tokens per CTA: a 64-wide K atom's MMAs (128 x n_tok x 64) per ~0.4 us of
  // issue steps; the widest tile for large batches
  pp.n_tok = T >= kPMaxN ? kPMaxN : ((T + 15) / 16) * 16;
  pp.t_tiles = (T + pp.n_tok - 1) / pp.n_tok;
  const int q_tiles = H_I;   // 128 features = one head per tile
  // two CTAs per SM when their stages fit twice in shared memory (small batches)
  const int slots = (2 * prolog_smem_bytes(pp.n_tok) <= 227 * 1024 ? 2 : 1) * num_sms;
  pp.split_q = split_for(q_tiles * pp.t_tiles, d_q / kPAtom, slots);
  pp.split_kw = split_for(2 * pp.t_tiles, d_model / kPAtom, slots);
  pp.q_bytes = (static_cast<size_t>(pp.split_q) * T * H_I * 128 * 4 + 255) / 256 * 256;
  pp.kw_bytes = (static_cast<size_t>(pp.split_kw) * T * 256 * 4 + 255) / 256 * 256;
  return pp;
}
}  // namespace

size_t prolog_workspace_bytes(int T, int H_I, int d_model, int d_q, int num_sms) {
  const PrologPlan pp = prolog_plan(T, H_I, d_model, d_q, num_sms);
  return pp.q_bytes + pp.kw_bytes;
}

cudaError_t launch_prolog(const SeqArgs& seq, const PrologArgs& a, void* workspace, const LaunchEnv& env,
                          std::string* plan, bool* unsupported, std::string* why) {
  *unsupported = false;
  if (seq.T == 0) {
    *plan += "prolog[empty]";
    return cudaSuccess;
  }
  const int T = seq.T;
  const int HD = a.H_I * 128;
  const PrologPlan pp = prolog_plan(T, a.H_I, a.d_model, a.d_q, env.num_sms);
  float* yq = static_cast<float*>(workspace);
  float* ykw = reinterpret_cast<float*>(static_cast<char*>(workspace) + pp.q_bytes);
  const int n_tok = pp.n_tok;
  const int t_tiles = pp.t_tiles;
  alignas(64) CUtensorMap wq_map, wk_map, ww_map, xq_map, x_map;
  if (!encode_tmap_2d(&wq_map, a.w_q, 2, a.d_q, HD, static_cast<uint64_t>(a.d_q) * 2, kPAtom, kPM, why) ||
      !encode_tmap_2d(&wk_map, a.w_k, 2, a.d_model, 128, static_cast<uint64_t>(a.d_model) * 2, kPAtom, kPM, why) ||
      !encode_tmap_2d(&ww_map, a.w_w, 2, a.d_model, a.H_I, static_cast<uint64_t>(a.d_model) * 2, kPAtom, kPM, why) ||
      !encode_tmap_2d(&xq_map, a.x_q, 2, a.d_q, T, static_cast<uint64_t>(a.d_q) * 2, kPAtom, n_tok, why) ||
      !encode_tmap_2d(&x_map, a.x, 2, a.d_model, T, static_cast<uint64_t>(a.d_model) * 2, kPAtom, n_tok, why)) {
    *unsupported = true;
    return cudaSuccess;
  }
  ProjParams p{};
  p.T = T;
  p.n_tok = n_tok;
  p.tmem_cols = n_tok <= 32 ? 32u : (n_tok <= 64 ? 64u : (n_tok <= 128 ? 128u : 256u));
  p.t_tiles = t_tiles;
  const int q_atoms = a.d_q / kPAtom, x_atoms = a.d_model / kPAtom;
  const int q_tiles = HD / kPM;
  // the key and head-weight tiles (the longer reductions) first in the grid
  const int64_t kw_slice = static_cast<int64_t>(T) * 256;
  p.job[1] = ProjJob{128, x_atoms, pp.split_kw, 1, 0, ykw, 256, kw_slice};
  p.job[2] = ProjJob{a.H_I, x_atoms, pp.split_kw, 1, t_tiles * pp.split_kw, ykw + 128, 256, kw_slice};
  p.job[0] = ProjJob{HD, q_atoms, pp.split_q, q_tiles, 2 * t_tiles * pp.split_kw, yq, HD,
                     static_cast<int64_t>(T) * HD};
  const int grid = p.job[0].first_cta + q_tiles * t_tiles * p.job[0].split;
  uint32_t dbg_withhold = 0;
  debug_wait_state(&p.wait_limit_ns, &dbg_withhold);
  const cudaError_t attr = ensure_smem_limit(reinterpret_cast<const void*>(prolog_proj_kernel),
                                             prolog_smem_bytes(kPMaxN), env.device);
  if (attr != cudaSuccess) return attr;
  cudaError_t e = launch_kernel(prolog_proj_kernel, dim3(grid), dim3(kPThreads), prolog_smem_bytes(n_tok), env.stream,
                                false, 1, wq_map, wk_map, ww_map, xq_map, x_map, p);
  if (e != cudaSuccess) return e;
  EpiParams ep{seq, a.H_I, yq, pp.split_q, ykw, pp.split_kw, a.gamma, a.beta, a.q_codes, a.q_scale, a.w,
               a.k_cache, a.k_scale};
  e = launch_kernel(prolog_epilogue_kernel, dim3(T, (a.H_I + kEpiHeads - 1) / kEpiHeads + 1), dim3(32 * kEpiHeads),
                    0, env.stream, true, 1, ep);
  if (e != cudaSuccess) return e;
  char buf[160];
  snprintf(buf, sizeof(buf), "prolog_proj[grid=%d,tok=%d,split=%d/%d]+prolog_epilogue", grid, n_tok,
           p.job[0].split, p.job[1].split);
  *plan += buf;
  return cudaGetLastError();
}

}  // namespace dsa
