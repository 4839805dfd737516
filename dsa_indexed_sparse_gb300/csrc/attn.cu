// Sparse MLA attention over the selected latent rows (step 3 of the DSA path).
//
// "Large Language Model Inference Acceleration in Practice", section 1.2 (SFA)
// and section 3.1: using the indices produced by the lightning indexer, the
// kernel reads only the selected positions' rows from the paged KV cache and runs
// flash attention over them.  MQA form over the MLA latent cache: each cache row
// holds a 576-d key (512 latent + 64 rope) whose first 512 values are also the
// value; all heads of a query share the rows.  For query t, head h and selected
// set S:
//     logit_s = scale * q[t,h] . row_s[0:576],  out = sum_s softmax(logit)_s row_s[0:512],
//     lse = log sum_s exp(logit_s).
//
// Kernels:
//  * attn_tc_kernel<kFp8> -- tensor-core path for H = 128, 512 + 64 dims, bf16 rows or
//    656-byte FP8 rows.  FP8 codes are widened to bf16 exactly (no scale applied)
//    while gathering; the per-row scale is applied to the latent part of the logit
//    (S_latent and S_rope accumulate in separate TMEM columns) and folded into P
//    for P V, so the FP8 path rounds nothing the bf16 path does not.  One CTA handles one
//    query, one half of the value dims (256 of 512) and one contiguous slice of the
//    selected rows.  The CTA pair covering both value halves computes the same
//    logits: O[128 x 512] fp32 would fill all of TMEM, so each CTA keeps a
//    [128 x 256] accumulator plus double-buffered logits.
//      warps 0-3: gather 32 selected rows per tile (lane = row: index -> page ->
//                 cache row) with 16-byte cp.async into a 128-byte-swizzled
//                 K-major tile; 4 tiles in flight (3 for FP8 rows);
//      warp 8   : issues S = Q K^T (M=128 heads, N=32 rows, K=576; the first 256
//                 query dims are read from TMEM, the rest from shared memory) and
//                 O += P V (M=128, N=256, K=32; P read from TMEM) with tcgen05.mma;
//      warps 4-7: online softmax, one thread per head (its TMEM lane), P written
//                 as bf16 into TMEM; the running max is only moved (and O
//                 rescaled in TMEM) when it grows by more than 2^8.
//  * attn_combine_kernel -- merges per-slice partial results by their LSE.
//  * attn_generic_kernel -- CUDA cores, any head count / dims / row format.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

DSA_DEFINE_STATUS_WORD(attn)

namespace dsa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// =============================================================== generic kernel
constexpr int kGenThreads = 128;

__device__ __forceinline__ float load_elem(MlaKind kind, const uint8_t* row, int d) {
  switch (kind) {
    case MlaKind::kF32:
      return reinterpret_cast<const float*>(row)[d];
    case MlaKind::kBF16:
      return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[d]);
    default: {  // 656-byte FP8 row
      if (d < 512) return e4m3_to_float(row[d]) * *reinterpret_cast<const float*>(row + 512);
      return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row + 528)[d - 512]);
    }
  }
}

__device__ __forceinline__ float block_reduce_max(float v, float* buf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  float r = buf[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, buf[w]);
  return r;
}
__device__ __forceinline__ float block_reduce_sum(float v, float* buf) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += buf[w];
  return r;
}

__global__ void __launch_bounds__(kGenThreads)
    attn_generic_kernel(SeqArgs seq, MlaArgs a) {
  grid_dep_wait();
  extern __shared__ float sm_gen[];
  const int dqk = a.d_latent + a.d_rope, dv = a.d_latent, K = a.K;
  float* qs = sm_gen;                                            // [dqk]
  float* ps = qs + dqk;                                          // [K] logits then weights
  int32_t* rows = reinterpret_cast<int32_t*>(ps + K);            // [K] physical rows
  __shared__ float red[kGenThreads / 32];
  const int h = blockIdx.x, t = blockIdx.y;
  const int qp = __ldg(seq.q_pos + t);
  const int b = __ldg(seq.q_seq + t);
  const bool q_ok = qp >= 0 && qp < seq.max_ctx && b >= 0 && b < seq.B;
  if (!q_ok && threadIdx.x == 0 && h == 0) atomicOr(&g_status_attn, kDevBadPos);
  const int64_t qoff = (static_cast<int64_t>(t) * a.H + h) * dqk;
  for (int d = threadIdx.x; d < dqk; d += blockDim.x) {
    qs[d] = (a.kind == MlaKind::kF32) ? static_cast<const float*>(a.q)[qoff + d]
                                      : bf16_bits_to_float(static_cast<const uint16_t*>(a.q)[qoff + d]);
  }
  __syncthreads();
  const uint8_t* kv = static_cast<const uint8_t*>(a.kv);
  const int32_t* bt = seq.block_table + static_cast<int64_t>(q_ok ? b : 0) * seq.bt_stride;
  float mloc = -INFINITY;
  for (int r = threadIdx.x; r < K; r += blockDim.x) {
    const int pos = __ldg(a.idx + static_cast<int64_t>(t) * K + r);
    int64_t prow = -1;
    if (q_ok && pos >= 0) {
      if (pos > qp) {
        atomicOr(&g_status_attn, kDevBadIndex);
      } else {
        prow = phys_row(bt, pos, seq.page_size, seq.n_pages, &g_status_attn);
      }
    }
    rows[r] = static_cast<int32_t>(prow);
    float logit = -INFINITY;
    if (prow >= 0) {
      const uint8_t* rp = kv + prow * a.row_bytes;
      float acc = 0.f;
      for (int d = 0; d < dqk; ++d) acc = fmaf(qs[d], load_elem(a.kind, rp, d), acc);
      logit = acc * a.softmax_scale;
    }
    ps[r] = logit;
    mloc = fmaxf(mloc, logit);
  }
  const float m = block_reduce_max(mloc, red);
  float lsum = 0.f;
  for (int r = threadIdx.x; r < K; r += blockDim.x) {
    const float p = (m == -INFINITY || ps[r] == -INFINITY) ? 0.f : __expf(ps[r] - m);
    ps[r] = p;
    lsum += p;
  }
  const float l = block_reduce_sum(lsum, red);  // includes a __syncthreads
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int64_t ooff = (static_cast<int64_t>(t) * a.H + h) * dv;
  for (int d = threadIdx.x; d < dv; d += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < K; ++r) {
      if (rows[r] >= 0) acc = fmaf(ps[r], load_elem(a.kind, kv + static_cast<int64_t>(rows[r]) * a.row_bytes, d), acc);
    }
    acc *= inv;
    if (a.kind == MlaKind::kF32)
      static_cast<float*>(a.out)[ooff + d] = acc;
    else
      static_cast<__nv_bfloat16*>(a.out)[ooff + d] = __float2bfloat16_rn(acc);
  }
  if (threadIdx.x == 0 && a.lse)
    a.lse[static_cast<int64_t>(t) * a.H + h] = l > 0.f ? m + logf(l) : -INFINITY;
}

// =============================================================== tcgen05 kernel
constexpr int kH = 128;          // heads = UMMA M
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;     // value dims per CTA = UMMA N of P V
constexpr int kBR = 32;          // rows per tile = UMMA N of Q K^T
constexpr int kTileBytes = kBR * kDqk * 2;         // 36864
constexpr int kThreads = 288;                      // 4 producer, 4 softmax, 1 MMA warp
constexpr int kProducerWarps = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescS = make_idesc(kFmtBF16, kFmtBF16, false, false, kH, kBR);
constexpr uint32_t kIdescPV = make_idesc(kFmtBF16, kFmtBF16, false, true, kH, kDvHalf);
constexpr float kRescaleThreshold = 8.0f;          // log2 units

// Shared memory and TMEM plan.  The first kQTmemDims query dims live in TMEM
// (A operand of Q K^T read from tensor memory), the rest in shared memory, and P
// lives in TMEM too, which leaves room for kStages gathered tiles.
//   TMEM columns: S [0,64) (two buffers), FP8 rope logits [64,128), P (16),
//   Q (kQTmemDims / 2), O [256, 512).
template <bool kFp8>
struct AttnCfg {
  static constexpr int kQTmemDims = kFp8 ? 192 : 256;
  static constexpr int kQTmemSteps = kQTmemDims / 16;
  static constexpr int kQSmemAtoms = (kDqk - kQTmemDims) / 64;
  static constexpr int kStages = kFp8 ? 3 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQSmemAtoms * kH * 128;
  static constexpr int kOffMask = kOffKV + kStages * kTileBytes;   // uint32 [stages]
  static constexpr int kOffScale = kOffMask + 16;                  // float [stages][32]
  static constexpr int kOffBar = kOffScale + kStages * kBR * 4;
  // barriers: full[S], empty[S], sfull[2], pfull, pvdone, ofull
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;          // tmem base, abort
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;          // + alignment slack
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColSr = 64;
  static constexpr uint32_t kColP = kFp8 ? 128 : 64;
  static constexpr uint32_t kColQ = kFp8 ? 160 : 128;
  static constexpr uint32_t kColO = 256;
  static_assert(kColQ + kQTmemDims / 2 <= kColO, "TMEM plan");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct TcAttnParams {
  SeqArgs seq;
  MlaArgs a;
  int32_t n_split;       // row slices per query
  int32_t rows_per_split;
  uint16_t* ws_o;        // [n_split, T, H, 512] bf16 partials (n_split > 1), each normalised by its own sum
  float* ws_lse;         // [n_split, T, H]
};

// Byte offset of 16-byte chunk `ch` of tile row `r` in a 128B-swizzled K-major
// tile of `rows` rows: atom (64 values) major, then row, then swizzled chunk.
__device__ __forceinline__ uint32_t sw128_offset(int r, int ch, int rows) {
  return static_cast<uint32_t>((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(TcAttnParams p) {
  using C = AttnCfg<kFp8>;
  grid_dep_wait();
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // re-aligned by pointer arithmetic on the shared array, so that the compiler
  // keeps every access through `sm` in the shared window
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* full = bars;          // [S] tile landed (32 producer lanes)
  uint64_t* empty = bars + S;     // [S] tile consumed by P V (MMA commit)
  uint64_t* sfull = bars + 2 * S; // [2] logits ready
  uint64_t* pfull = bars + 2 * S + 2;
  uint64_t* pvdone = bars + 2 * S + 3;
  uint64_t* ofull = bars + 2 * S + 4;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile uint32_t* mask_s = reinterpret_cast<volatile uint32_t*>(sm + C::kOffMask);
  volatile float* row_scale = reinterpret_cast<volatile float*>(sm + C::kOffScale);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x & 1;                     // value half
  const int rest = blockIdx.x >> 1;
  const int split = rest % p.n_split;
  const int t = p.seq.T - 1 - rest / p.n_split;   // last query first (longest causal history)
  const int K = p.a.K;
  const int r0 = split * p.rows_per_split;
  const int r1 = min(K, r0 + p.rows_per_split);
  const int ntiles = (r1 - r0 + kBR - 1) / kBR;     // >= 1 (host guarantees r0 < K)

  int qp = __ldg(p.seq.q_pos + t);
  int b = __ldg(p.seq.q_seq + t);
  if (qp < 0 || qp >= p.seq.max_ctx || b < 0 || b >= p.seq.B) {
    if (threadIdx.x == 0) atomicOr(&g_status_attn, kDevBadPos);
    qp = -1;  // every row masked
    b = 0;
  }
  const uint16_t* qg = static_cast<const uint16_t*>(p.a.q) + static_cast<int64_t>(t) * kH * kDqk;

  // ---- setup: barriers, TMEM, Q (shared-memory part via cp.async) -----------
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 32);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&sfull[i], 1);
    mbar_init(pfull, 128);
    mbar_init(pvdone, 1);
    mbar_init(ofull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(misc, kTmemCols);
    tmem_relinquish();
  }
  {
    const uint32_t qbase = smem_u32(sm + C::kOffQ);
    constexpr int kChunks = (kDqk - C::kQTmemDims) / 8;  // 16-byte chunks per row in smem
    for (int i = threadIdx.x; i < kH * kChunks; i += kThreads) {
      const int h = i / kChunks, ch = i % kChunks;
      cp_async16(qbase + sw128_offset(h, ch, kH), qg + h * kDqk + C::kQTmemDims + ch * 8);
    }
    cp_async_commit();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (warp >= 4 && warp < 8) {
    // Q dims [0, kQTmemDims) of head h -> TMEM lane h (two bf16 per column)
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint4* qrow = reinterpret_cast<const uint4*>(qg + h * kDqk);
#pragma unroll 1
    for (int blk = 0; blk < C::kQTmemDims / 64; ++blk) {
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(qrow + blk * 8 + i);
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
      }
      tmem_st32(tmem + lane_off + C::kColQ + blk * 32, r);
    }
    tmem_st_wait();
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < kProducerWarps) {
    // ------------------------------------------------ producers: warp w < S owns stage w and
    // loads its tiles j = w mod S.  (A stage's empty barrier must be waited on by
    // one warp in phase order: a warp waiting two phases ahead of the barrier's
    // pending phase would see that parity as completed and overwrite a tile in use.)
    const uint8_t* kv = static_cast<const uint8_t*>(p.a.kv);
    const int32_t* bt = p.seq.block_table + static_cast<int64_t>(b) * p.seq.bt_stride;
    const int32_t* idx = p.a.idx + static_cast<int64_t>(t) * K;
    for (int j = warp; warp < S && j < ntiles; j += S) {
      const int st = j % S;
      // lane r resolves tile row r (index -> page -> cache row) before the wait
      int64_t my_row = -1;
      float my_scale = 0.f;
      const int gi = r0 + j * kBR + lane;
      if (gi < r1) {
        const int pos = __ldg(idx + gi);
        if (pos >= 0) {
          if (pos > qp)
            atomicOr(&g_status_attn, kDevBadIndex);
          else
            my_row = phys_row(bt, pos, p.seq.page_size, p.seq.n_pages, &g_status_attn);
        }
      }
      if (kFp8 && my_row >= 0)
        my_scale = __ldg(reinterpret_cast<const float*>(kv + my_row * p.a.row_bytes + 512));
      if (j >= S) {
        const bool ok = mbar_wait(&empty[st], ((j / S) - 1) & 1, &g_status_attn, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const uint32_t stage = smem_u32(sm + C::kOffKV + st * kTileBytes);
      const uint32_t bits = __ballot_sync(0xffffffffu, my_row >= 0);
      if (kFp8) row_scale[st * kBR + lane] = my_scale;
      if (lane == 0) mask_s[st] = bits;
      if (!kFp8) {
        // 72 16-byte chunks per row; consecutive lanes take consecutive chunks
#pragma unroll 4
        for (int i = lane; i < kBR * (kDqk / 8); i += 32) {
          const int rr = i / (kDqk / 8), ch = i % (kDqk / 8);
          const int64_t prow = __shfl_sync(0xffffffffu, my_row, rr);
          if (prow >= 0)
            cp_async16(stage + sw128_offset(rr, ch, kBR), kv + prow * p.a.row_bytes + ch * 16);
          else
            st_shared_v4(stage + sw128_offset(rr, ch, kBR), 0u, 0u, 0u, 0u);
        }
      } else {
        // latent: 16 e4m3 codes per lane and row, 8 rows' loads in flight before
        // any conversion; widened to bf16 exactly (two 16-byte chunks); rope by cp.async
#pragma unroll 1
        for (int r8 = 0; r8 < kBR; r8 += 8) {
          uint4 raw[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int64_t prow = __shfl_sync(0xffffffffu, my_row, r8 + q);
            raw[q] = prow >= 0 ? ld_global_nc_v4(kv + prow * p.a.row_bytes + lane * 16) : make_uint4(0, 0, 0, 0);
            if (lane < 8) {
              if (prow >= 0)
                cp_async16(stage + sw128_offset(r8 + q, 64 + lane, kBR), kv + prow * p.a.row_bytes + 528 + lane * 16);
              else
                st_shared_v4(stage + sw128_offset(r8 + q, 64 + lane, kBR), 0u, 0u, 0u, 0u);
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
            uint32_t o[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w[k] & 0xFFFFu));
              const float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w[k] >> 16));
              o[2 * k] = pack_bf16x2(lo.x, lo.y);
              o[2 * k + 1] = pack_bf16x2(hi.x, hi.y);
            }
            st_shared_v4(stage + sw128_offset(r8 + q, 2 * lane, kBR), o[0], o[1], o[2], o[3]);
            st_shared_v4(stage + sw128_offset(r8 + q, 2 * lane + 1, kBR), o[4], o[5], o[6], o[7]);
          }
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(&full[st]);
    }
  } else if (warp == 8) {
    // ------------------------------------------------ MMA issuer (whole warp, elected lane issues)
    // Descriptors are built once; the unrolled issue loops only add constant byte
    // offsets (>> 4) to the start-address field, and one elected lane issues a
    // whole block of MMAs (this keeps the issue cost near 30-40 cycles per MMA).
    const uint64_t dq0 = make_sdesc(smem_u32(sm + C::kOffQ), 16, 1024, kLayoutSw128);
    const uint64_t dk0 = make_sdesc(smem_u32(sm + C::kOffKV), 16, 1024, kLayoutSw128);
    const uint64_t dv0 = make_sdesc(smem_u32(sm + C::kOffKV) + c * 4 * kBR * 128, kBR * 128, 1024, kLayoutSw128);
    auto issue_pv = [&](int j) {
      const uint64_t dv = dv0 + static_cast<uint64_t>(((j % S) * kTileBytes) >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kBR / 16; ++kk)
          umma_f16_tmem_a(tmem + C::kColO, tmem + C::kColP + kk * 8, dv + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                          kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pvdone);
        umma_commit(&empty[j % S]);
      }
      __syncwarp();
    };
    // Issue S_j as soon as tile j has landed (and its S buffer is free, i.e.
    // P_{j-2} was consumed) and P V_j as soon as P_j is written, in whichever
    // order they become ready, so neither kind of MMA waits on the other's inputs.
    int next_s = 0, next_pv = 0;
    uint32_t spins = 0;
    uint64_t stall_t0 = 0;
    while (next_pv < ntiles) {
      bool progress = false;
      const bool s_ready = next_s < ntiles && next_s <= next_pv + 1 &&
                           mbar_test_wait(smem_u32(&full[next_s % S]), (next_s / S) & 1);
      if (__shfl_sync(0xffffffffu, s_ready, 0)) {
        tc_fence_after();
        const int j = next_s;
        const uint64_t dk = dk0 + static_cast<uint64_t>(((j % S) * kTileBytes) >> 4);
        const uint32_t col_s = tmem + C::kColS + (j & 1) * kBR;
        const uint32_t col_r = tmem + C::kColSr + (j & 1) * kBR;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kDqk / 16; ++kk) {
            const uint64_t db = dk + static_cast<uint64_t>(((kk >> 2) * kBR * 128 + (kk & 3) * 32) >> 4);
            // FP8 rows: latent (k < 512) and rope (k >= 512) logits in separate columns
            const bool rope = kFp8 && kk >= kDv / 16;
            const uint32_t acc = (kk == 0 || (kFp8 && kk == kDv / 16)) ? 0u : 1u;
            if (kk < C::kQTmemSteps) {
              umma_f16_tmem_a(rope ? col_r : col_s, tmem + C::kColQ + kk * 8, db, kIdescS, acc);
            } else {
              const int qk = kk - C::kQTmemSteps;
              const uint64_t da = dq0 + static_cast<uint64_t>(((qk >> 2) * kH * 128 + (qk & 3) * 32) >> 4);
              umma_f16(rope ? col_r : col_s, da, db, kIdescS, acc);
            }
          }
          umma_commit(&sfull[j & 1]);
        }
        __syncwarp();
        ++next_s;
        progress = true;
      }
      const bool p_ready = next_pv < next_s && mbar_test_wait(smem_u32(pfull), next_pv & 1);
      if (__shfl_sync(0xffffffffu, p_ready, 0)) {
        tc_fence_after();
        issue_pv(next_pv);
        if (next_pv == ntiles - 1) {
          if (elect_one()) umma_commit(ofull);
          __syncwarp();
        }
        ++next_pv;
        progress = true;
      }
      if (progress) {
        stall_t0 = 0;
      } else if ((++spins & 63u) == 0u) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
        const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
        if (stall_t0 == 0) {
          stall_t0 = now;
        } else if (now - stall_t0 > kWaitLimitNs) {
          if (lane == 0) {
            atomicOr(&g_status_attn, kDevTimeout);
            *abort_flag = 1;
          }
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 4-7)
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.a.softmax_scale * kLog2e;
    // l: sum of the bf16 weights actually multiplied into O (normalising by it
    // makes the output an exact convex combination of the rows); l32: the same
    // weights in fp32, for the log-sum-exp.
    float m = -INFINITY, l = 0.f, l32 = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % S;
      ok = mbar_wait(&sfull[j & 1], (j >> 1) & 1, &g_status_attn, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // The producer's mask and scales are ordered by its release on full[st]:
      // that phase is still the current one here (the stage is only refilled
      // after this tile's P V, which needs this thread's arrival on pfull).
      ok = mbar_wait(&full[st], (j / S) & 1, &g_status_attn, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + C::kColS + (j & 1) * kBR, r);
      const uint32_t vmask = mask_s[st];
      float x[32];
      float mloc = -INFINITY;
      if (kFp8) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + C::kColSr + (j & 1) * kBR, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float lg = fmaf(row_scale[st * kBR + i], __uint_as_float(r[i]), __uint_as_float(rr[i]));
          x[i] = ((vmask >> i) & 1u) ? lg * sl2 : -INFINITY;
          mloc = fmaxf(mloc, x[i]);
        }
      } else {
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = ((vmask >> i) & 1u) ? __uint_as_float(r[i]) * sl2 : -INFINITY;
          mloc = fmaxf(mloc, x[i]);
        }
      }
      if (j >= 1) {
        // P V_{j-1} must have read P (TMEM) and written O before P and O change
        ok = mbar_wait(pvdone, (j - 1) & 1, &g_status_attn, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const float m_new = fmaxf(m, mloc);
      const bool need = m_new > m + kRescaleThreshold;
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        const float f = need ? exp2f(m - m_new) : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kDvHalf / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + C::kColO + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tmem + lane_off + C::kColO + cc * 32, o);
        }
      }
      if (need) {
        const float f = exp2f(m - m_new);
        l *= f;
        l32 *= f;
        m = m_new;
      }
      const float msub = (m == -INFINITY) ? 0.f : m;
      float psum = 0.f, psum32 = 0.f;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = fast_exp2(x[2 * i] - msub), p1 = fast_exp2(x[2 * i + 1] - msub);
        psum32 += p0 + p1;
        if (kFp8) {
          // P V runs on the unscaled codes: fold the row scale into P; the
          // denominator takes the rounded weights divided back by the scale
          const float s0 = row_scale[st * kBR + 2 * i], s1 = row_scale[st * kBR + 2 * i + 1];
          __nv_bfloat162 v = __floats2bfloat162_rn(p0 * s0, p1 * s1);
          pk[i] = *reinterpret_cast<uint32_t*>(&v);
          const float2 back = __bfloat1622float2(v);
          psum += (s0 > 0.f ? back.x / s0 : 0.f) + (s1 > 0.f ? back.y / s1 : 0.f);
        } else {
          __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
          pk[i] = *reinterpret_cast<uint32_t*>(&v);
          const float2 back = __bfloat1622float2(v);
          psum += back.x + back.y;
        }
      }
      l += psum;
      l32 += psum32;
      tmem_st16(tmem + lane_off + C::kColP, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pfull);
    }
    if (ok) {
      ok = mbar_wait(ofull, 0, &g_status_attn, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l32 > 0.f ? (m + log2f(l32)) * kLn2 : -INFINITY;
      const int64_t th = static_cast<int64_t>(t) * kH + h;
      // all MMAs are complete (ofull), so the stage buffers are idle: 4 KB per warp
      const uint32_t stg = smem_u32(sm + C::kOffKV) + quarter * 4096;
      const int64_t th0 = static_cast<int64_t>(t) * kH + quarter * 32;   // this warp's first head
      // bf16 rows of this warp's 32 heads: the output, or this slice's partial
      // (normalised by its own sum; the combine weights it by its LSE)
      const bool part = p.n_split > 1;
      const int64_t row0 = part ? static_cast<int64_t>(split) * p.seq.T * kH + th0 : th0;
      uint8_t* out = reinterpret_cast<uint8_t*>(part ? p.ws_o : static_cast<uint16_t*>(p.a.out)) +
                     (row0 * kDv + c * kDvHalf) * 2;
#pragma unroll 1
      for (int cc = 0; cc < kDvHalf / 64; ++cc) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + C::kColO + cc * 64, o0);
        tmem_ld32(tmem + lane_off + C::kColO + cc * 64 + 32, o1);
        tmem_ld_wait();
        uint32_t pk2[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pk2[i] = pack_bf16x2(__uint_as_float(o0[2 * i]) * inv, __uint_as_float(o0[2 * i + 1]) * inv);
          pk2[16 + i] = pack_bf16x2(__uint_as_float(o1[2 * i]) * inv, __uint_as_float(o1[2 * i + 1]) * inv);
        }
        warp_store_rows128(stg, pk2, out + cc * 128, kDv * 2, lane);
      }
      if (part) {
        if (c == 0) p.ws_lse[static_cast<int64_t>(split) * p.seq.T * kH + th] = lse;
      } else if (c == 0 && p.a.lse) {
        p.a.lse[th] = lse;
      }
    }
  }

  grid_dep_launch();  // this CTA's work is done: the next kernel may launch
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// bf16 rows, 48-row tiles, three stages.
//
// Producers (warps 0-11): three groups of four warps own one stage each and
// load every third tile (12 rows per warp; a warp issues cp.async copies at
// ~30 ns per instruction here, so the warps per tile set how fast it lands).  Lanes resolve the rows (index -> page
// -> cache row) as soon as the group's previous tile has landed and ask L2 to
// fetch them; once the stage is free every lane copies its fixed 16-byte
// chunks of each row with cp.async into the 128B-swizzled K-major tile; rows
// that select nothing are zeroed.  (On this GPU a tile::gather4 TMA producer
// reached ~12 GB/s per SM and cp.async gathers ~60 GB/s.)
//
// MMA warps: warp 12 issues Q K^T_{j+1} (N = 48 rows) as soon as the softmax
// has read S_j and tile j+1 has landed, so it runs during the softmax of tile
// j; warp 13 issues P V_j (N = 256 value dims, P read from TMEM) as soon as P_j
// is written.  (One warp issuing both made a ready P V wait behind the issue
// of a Q K^T and vice versa: the issuing thread blocks until the tensor pipe
// has taken the instructions.)  An M=128
// K=16 step whose A operand (the query) sits in shared memory reads 6 KB of
// shared memory and takes ~53 clk, one with A in TMEM ~36 clk, so the first 320
// query dims live in TMEM.
//
// Softmax (warps 14-17): one thread per head (its TMEM lane), 48 logits a tile,
// running max moved (and O rescaled in TMEM) only when it grows by more than
// 2^8.
//
// TMEM: S [0,48), P [64,88), Q [96,256), O [256,512).  Shared memory: query
// dims [320, 576) (64 KB) + three 54 KB tiles.  (A dedicated MMA warp issuing
// Q K^T_{j+1} during softmax_j hides the softmax; the third stage hides the
// gather of a tile behind the work on the other two.)
constexpr int kBR48 = 48;
constexpr int kTile48Bytes = kBR48 * kDqk * 2;                 // 55296
constexpr int kT48Stages = 3;
constexpr int kT48QTmemDims = 320;
constexpr int kT48QTmemSteps = kT48QTmemDims / 16;             // 20
constexpr int kT48QSmemAtoms = (kDqk - kT48QTmemDims) / 64;    // 4
constexpr int kT48OffQ = 0;
constexpr int kT48OffKV = kT48QSmemAtoms * kH * 128;           // 65536
constexpr int kT48OffMask = kT48OffKV + kT48Stages * kTile48Bytes;  // uint16 [stages][4]
constexpr int kT48OffBar = kT48OffMask + kT48Stages * 4 * 2 + 8;
// barriers: full[3], empty[3], sfull, sfree, pfull, pvdone, ofull
constexpr int kT48NumBars = 2 * kT48Stages + 5;
constexpr int kT48OffMisc = kT48OffBar + kT48NumBars * 8;
constexpr int kT48Used = kT48OffMisc + 16;                     // bytes used from the aligned base
// the dynamic shared-memory base is re-aligned to 1024 B inside the kernel; this
// much slack is requested for it (the kernel checks that it sufficed)
constexpr int kT48Slack = 232448 - kT48Used;
constexpr int kT48SmemBytes = kT48Used + kT48Slack;
constexpr int kT48Threads = 576;   // warps 0-11 producers, 12 Q K^T, 13 P V, 14-17 softmax
constexpr int kT48Mma = 12;        // Q K^T issuer; also allocates TMEM
constexpr int kT48Pv = 13;         // P V issuer
constexpr int kT48Soft = 14;       // first softmax warp
constexpr int kT48Producers = 4;   // warps per stage group
constexpr uint32_t kT48ColS = 0, kT48ColP = 64, kT48ColQ = 96, kT48ColO = 256;
constexpr uint32_t kIdescS48 = make_idesc(kFmtBF16, kFmtBF16, false, false, kH, kBR48);
static_assert(kT48ColQ + kT48QTmemDims / 2 <= kT48ColO, "TMEM plan");
static_assert(kT48ColP + kBR48 / 2 <= kT48ColQ && kT48ColS + kBR48 <= kT48ColP, "TMEM plan");
static_assert(kT48Slack >= 128, "shared memory budget");

// Q K^T of one 48-row tile (elected lane of the MMA warp).
__device__ __forceinline__ void t48_issue_s(uint32_t tmem, uint64_t dq0, uint64_t dk) {
#pragma unroll
  for (int kk = 0; kk < kDqk / 16; ++kk) {
    const uint64_t db = dk + static_cast<uint64_t>(((kk >> 2) * kBR48 * 128 + (kk & 3) * 32) >> 4);
    const uint32_t acc = kk == 0 ? 0u : 1u;
    if (kk < kT48QTmemSteps) {
      umma_f16_tmem_a(tmem + kT48ColS, tmem + kT48ColQ + kk * 8, db, kIdescS48, acc);
    } else {
      const int qk = kk - kT48QTmemSteps;
      const uint64_t da = dq0 + static_cast<uint64_t>(((qk >> 2) * kH * 128 + (qk & 3) * 32) >> 4);
      umma_f16(tmem + kT48ColS, da, db, kIdescS48, acc);
    }
  }
}

__global__ void __launch_bounds__(kT48Threads, 1) attn_tc48_kernel(TcAttnParams p) {
  grid_dep_wait();
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // re-aligned by pointer arithmetic on the shared array, so that the compiler
  // keeps every access through `sm` in the shared window
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  if (sm - sm_raw > kT48Slack) {   // block-uniform: the re-aligned layout would not fit
    if (threadIdx.x == 0) atomicOr(&g_status_attn, kDevTimeout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kT48OffBar);
  uint64_t* full = bars;            // [3] tile landed (one arrival per warp of the stage's group)
  uint64_t* empty = bars + 3;       // [3] tile consumed by P V
  uint64_t* sfull = bars + 6;       // logits ready
  uint64_t* sfree = bars + 7;       // logits read by the softmax (S buffer reusable)
  uint64_t* pfull = bars + 8;
  uint64_t* pvdone = bars + 9;
  uint64_t* ofull = bars + 10;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + kT48OffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile uint16_t* mask16 = reinterpret_cast<volatile uint16_t*>(sm + kT48OffMask);   // [stage][warp]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x & 1;
  const int rest = blockIdx.x >> 1;
  const int split = rest % p.n_split;
  const int t = p.seq.T - 1 - rest / p.n_split;   // last query first (longest causal history)
  const int K = p.a.K;
  const int r0 = split * p.rows_per_split;
  const int r1 = min(K, r0 + p.rows_per_split);
  const int ntiles = (r1 - r0 + kBR48 - 1) / kBR48;

  int qp = __ldg(p.seq.q_pos + t);
  int b = __ldg(p.seq.q_seq + t);
  if (qp < 0 || qp >= p.seq.max_ctx || b < 0 || b >= p.seq.B) {
    if (threadIdx.x == 0) atomicOr(&g_status_attn, kDevBadPos);
    qp = -1;
    b = 0;
  }
  const uint16_t* qg = static_cast<const uint16_t*>(p.a.q) + static_cast<int64_t>(t) * kH * kDqk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kT48Stages; ++i) {
      mbar_init(&full[i], kT48Producers);
      mbar_init(&empty[i], 1);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, 128);
    mbar_init(pfull, 128);
    mbar_init(pvdone, 1);
    mbar_init(ofull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kT48Mma) {
    tmem_alloc(misc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  // The producers start gathering tiles at once; warps 12-17 stage the query
  // meanwhile (dims [320, 576) in shared memory, [0, 320) in TMEM) and meet at
  // named barrier 1 before the first MMA.
  constexpr uint32_t kQBar = 1, kQBarThreads = 6 * 32;
  if (warp >= kT48Mma) {
    const uint32_t qbase = smem_u32(sm + kT48OffQ);
    constexpr int kChunks = (kDqk - kT48QTmemDims) / 8;
    for (int i = threadIdx.x - kT48Mma * 32; i < kH * kChunks; i += kQBarThreads) {
      const int h = i / kChunks, ch = i % kChunks;
      cp_async16(qbase + sw128_offset(h, ch, kH), qg + h * kDqk + kT48QTmemDims + ch * 8);
    }
    cp_async_commit();
  }
  if (warp >= kT48Soft) {
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint4* qrow = reinterpret_cast<const uint4*>(qg + h * kDqk);
#pragma unroll 1
    for (int blk = 0; blk < kT48QTmemDims / 64; ++blk) {
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = __ldg(qrow + blk * 8 + i);
        r[4 * i] = v.x;
        r[4 * i + 1] = v.y;
        r[4 * i + 2] = v.z;
        r[4 * i + 3] = v.w;
      }
      tmem_st32(tmem + lane_off + kT48ColQ + blk * 32, r);
    }
    tmem_st_wait();
  }
  if (warp >= kT48Mma) {
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_sync(kQBar, kQBarThreads);
    tc_fence_after();
  }

  if (warp < kT48Mma) {
    // ------------------------------------------------ producers: group g = warp / 4 loads tiles
    // j = g mod 3 into stage g; warp w = warp % 4 copies tile rows [12w, 12w+12)
    constexpr int kRows = kBR48 / kT48Producers;
    const int grp = warp / kT48Producers, pw = warp % kT48Producers;
    const uint8_t* kv = static_cast<const uint8_t*>(p.a.kv);
    const int32_t* bt = p.seq.block_table + static_cast<int64_t>(b) * p.seq.bt_stride;
    const int32_t* idx = p.a.idx + static_cast<int64_t>(t) * K;
    // this lane's 16-byte chunks of a row: ch = lane, lane + 32, and lane + 64 for lanes < 8
    const int nch = lane < 8 ? 3 : 2;
    uint32_t dst_off[3], src_off[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int ch = lane + 32 * k;
      dst_off[k] = static_cast<uint32_t>((ch >> 3) * kBR48 * 128);   // atom block
      src_off[k] = static_cast<uint32_t>(ch * 16);
    }
    const int st = grp;
    const uint32_t stage = smem_u32(sm + kT48OffKV + st * kTile48Bytes);
    for (int j = grp; j < ntiles; j += kT48Stages) {
      int64_t my_row = -1;
      if (lane < kRows) {
        const int gi = r0 + j * kBR48 + pw * kRows + lane;
        if (gi < r1) {
          const int pos = __ldg(idx + gi);
          if (pos >= 0) {
            if (pos > qp)
              atomicOr(&g_status_attn, kDevBadIndex);
            else
              my_row = phys_row(bt, pos, p.seq.page_size, p.seq.n_pages, &g_status_attn);
          }
        }
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, my_row >= 0) & ((1u << kRows) - 1u);
      if (j >= kT48Stages) {
        // the stage is still busy: have L2 fetch this warp's rows (9 lines of 128 B each) meanwhile
#pragma unroll
        for (int k = 0; k < (kRows * 9 + 31) / 32; ++k) {
          const int i = lane + 32 * k;
          const int64_t prow = __shfl_sync(0xffffffffu, my_row, min(i / 9, kRows - 1));
          if (i < kRows * 9 && prow >= 0) prefetch_l2(kv + prow * p.a.row_bytes + (i % 9) * 128);
        }
        const bool ok = mbar_wait(&empty[st], ((j / kT48Stages) - 1) & 1, &g_status_attn, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) mask16[st * 4 + pw] = static_cast<uint16_t>(bits);
      // every row number first: a shuffle queues behind earlier cp.async copies
      int32_t rows[kRows];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) rows[rr] = __shfl_sync(0xffffffffu, static_cast<int32_t>(my_row), rr);
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        const int r = pw * kRows + rr;                       // row within the tile
        const int64_t prow = rows[rr];
        const uint32_t drow = stage + static_cast<uint32_t>(r * 128);
        if (prow >= 0) {
          const uint8_t* srow = kv + prow * p.a.row_bytes;
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            if (k < nch) {
              const uint32_t sw = static_cast<uint32_t>((((lane + 32 * k) & 7) ^ (r & 7)) << 4);
              cp_async16(drow + dst_off[k] + sw, srow + src_off[k]);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            if (k < nch) {
              const uint32_t sw = static_cast<uint32_t>((((lane + 32 * k) & 7) ^ (r & 7)) << 4);
              st_shared_v4(drow + dst_off[k] + sw, 0u, 0u, 0u, 0u);
            }
          }
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
    }
  } else if (warp == kT48Mma || warp == kT48Pv) {
    // ------------------------------------------------ MMA issuers (whole warp, elected lane issues)
    // Bounded polls on the non-suspending test_wait: these waits are on the
    // critical path of every tile.
    auto poll = [&](uint64_t* bar, uint32_t parity) -> bool {
      const uint32_t addr = smem_u32(bar);
      uint64_t t0 = 0;
      for (uint32_t it = 0;; ++it) {
        if (__shfl_sync(0xffffffffu, mbar_test_wait(addr, parity) ? 1 : 0, 0)) return true;
        if ((it & 255u) == 255u) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) return false;
          const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > kWaitLimitNs) {
            if (lane == 0) {
              atomicOr(&g_status_attn, kDevTimeout);
              *abort_flag = 1;
            }
            return false;
          }
        }
      }
    };
    if (warp == kT48Mma) {
      const uint64_t dq0 = make_sdesc(smem_u32(sm + kT48OffQ), 16, 1024, kLayoutSw128);
      const uint64_t dk0 = make_sdesc(smem_u32(sm + kT48OffKV), 16, 1024, kLayoutSw128);
      for (int j = 0; j < ntiles; ++j) {
        // Q K^T_j: tile j has landed and the softmax has read S_{j-1}
        if (j >= 1 && !poll(sfree, (j - 1) & 1)) break;
        if (!poll(&full[j % kT48Stages], (j / kT48Stages) & 1)) break;
        tc_fence_after();
        if (elect_one()) {
          t48_issue_s(tmem, dq0, dk0 + static_cast<uint64_t>(((j % kT48Stages) * kTile48Bytes) >> 4));
          umma_commit(sfull);
        }
        __syncwarp();
      }
    } else {
      const uint64_t dv0 = make_sdesc(smem_u32(sm + kT48OffKV) + c * 4 * kBR48 * 128, kBR48 * 128, 1024, kLayoutSw128);
      for (int j = 0; j < ntiles; ++j) {
        // P V_j as soon as P_j is written.  Its commits also cover Q K^T_j (complete
        // before the softmax wrote P_j), so empty[st] frees the whole stage and
        // ofull marks every MMA of the CTA done.
        if (!poll(pfull, j & 1)) break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>(((j % kT48Stages) * kTile48Bytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBR48 / 16; ++kk)
            umma_f16_tmem_a(tmem + kT48ColO, tmem + kT48ColP + kk * 8, dv + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                            kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(pvdone);
          umma_commit(&empty[j % kT48Stages]);
          if (j == ntiles - 1) umma_commit(ofull);
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 14-17)
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.a.softmax_scale * kLog2e;
    float m = -INFINITY, l = 0.f, l32 = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kT48Stages;
      ok = mbar_wait(sfull, j & 1, &g_status_attn, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // the producers' row mask is ordered by their release on full[st] (still the
      // current phase: the stage is refilled only after this tile's P V)
      ok = mbar_wait(&full[st], (j / kT48Stages) & 1, &g_status_attn, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s0[32], s1[16];
      tmem_ld32(tmem + lane_off + kT48ColS, s0);
      tmem_ld16(tmem + lane_off + kT48ColS + 32, s1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(sfree);
      uint64_t vmask = 0;
#pragma unroll
      for (int w = 0; w < kT48Producers; ++w)
        vmask |= static_cast<uint64_t>(mask16[st * 4 + w]) << (w * (kBR48 / kT48Producers));
      float x[kBR48];
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBR48; ++i) {
        const uint32_t raw = i < 32 ? s0[i & 31] : s1[(i - 32) & 15];
        x[i] = ((vmask >> i) & 1u) ? __uint_as_float(raw) * sl2 : -INFINITY;
        mloc = fmaxf(mloc, x[i]);
      }
      if (j >= 1) {
        // P V_{j-1} has read P and written O
        ok = mbar_wait(pvdone, (j - 1) & 1, &g_status_attn, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const float m_new = fmaxf(m, mloc);
      const bool need = m_new > m + kRescaleThreshold;
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        const float f = need ? exp2f(m - m_new) : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kDvHalf / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + kT48ColO + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tmem + lane_off + kT48ColO + cc * 32, o);
        }
      }
      if (need) {
        const float f = exp2f(m - m_new);
        l *= f;
        l32 *= f;
        m = m_new;
      }
      const float msub = (m == -INFINITY) ? 0.f : m;
      float psum = 0.f, psum32 = 0.f;
      uint32_t pk[kBR48 / 2];
#pragma unroll
      for (int i = 0; i < kBR48 / 2; ++i) {
        const float p0 = fast_exp2(x[2 * i] - msub), p1 = fast_exp2(x[2 * i + 1] - msub);
        psum32 += p0 + p1;
        __nv_bfloat162 v = __floats2bfloat162_rn(p0, p1);
        pk[i] = *reinterpret_cast<uint32_t*>(&v);
        const float2 back = __bfloat1622float2(v);
        psum += back.x + back.y;
      }
      l += psum;
      l32 += psum32;
      {
        uint32_t pa[16], pb[8];
#pragma unroll
        for (int i = 0; i < 16; ++i) pa[i] = pk[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) pb[i] = pk[16 + i];
        tmem_st16(tmem + lane_off + kT48ColP, pa);
        tmem_st8(tmem + lane_off + kT48ColP + 16, pb);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(pfull);
    }
    if (ok) {
      ok = mbar_wait(ofull, 0, &g_status_attn, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l32 > 0.f ? (m + log2f(l32)) * kLn2 : -INFINITY;
      const int64_t th = static_cast<int64_t>(t) * kH + h;
      // all MMAs are complete (ofull), so the stage buffers are idle: 4 KB per warp
      const uint32_t stg = smem_u32(sm + kT48OffKV) + quarter * 4096;
      const int64_t th0 = static_cast<int64_t>(t) * kH + quarter * 32;   // this warp's first head
      // bf16 rows of this warp's 32 heads: the output, or this slice's partial
      // (normalised by its own sum; the combine weights it by its LSE)
      const bool part = p.n_split > 1;
      const int64_t row0 = part ? static_cast<int64_t>(split) * p.seq.T * kH + th0 : th0;
      uint8_t* out = reinterpret_cast<uint8_t*>(part ? p.ws_o : static_cast<uint16_t*>(p.a.out)) +
                     (row0 * kDv + c * kDvHalf) * 2;
#pragma unroll 1
      for (int cc = 0; cc < kDvHalf / 64; ++cc) {
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + kT48ColO + cc * 64, o0);
        tmem_ld32(tmem + lane_off + kT48ColO + cc * 64 + 32, o1);
        tmem_ld_wait();
        uint32_t pk2[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          pk2[i] = pack_bf16x2(__uint_as_float(o0[2 * i]) * inv, __uint_as_float(o0[2 * i + 1]) * inv);
          pk2[16 + i] = pack_bf16x2(__uint_as_float(o1[2 * i]) * inv, __uint_as_float(o1[2 * i + 1]) * inv);
        }
        warp_store_rows128(stg, pk2, out + cc * 128, kDv * 2, lane);
      }
      if (part) {
        if (c == 0) p.ws_lse[static_cast<int64_t>(split) * p.seq.T * kH + th] = lse;
      } else if (c == 0 && p.a.lse) {
        p.a.lse[th] = lse;
      }
    }
  }

  grid_dep_launch();  // this CTA's work is done: the next kernel may launch
  tc_fence_before();
  __syncthreads();
  if (warp == kT48Mma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merges row slices: out[t,h,:] = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max_s lse_s);
// lse = max + log sum_s w_s.  The partials O_s are bf16 rows, each normalised by
// its own slice's sum.  One CTA of two warps per (query, pair of heads); a warp per
// head, each lane owning 16 value dims (two 16-byte vectors per slice).  Slices go
// in batches of 16 whose row loads and LSE loads are all in flight together (one
// L2 round trip per batch), merged with a running maximum across batches.
constexpr int kCombineHeads = 2;
constexpr int kCombineBatch = 16;
__global__ void __launch_bounds__(32 * kCombineHeads)
    attn_combine_kernel(const uint16_t* ws_o, const float* ws_lse, int n_split, int T,
                        __nv_bfloat16* out, float* lse_out) {
  grid_dep_wait();
  constexpr int H = kH;
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kCombineHeads + warp;
  const int64_t th = static_cast<int64_t>(t) * H + h;
  const int64_t slice_stride = static_cast<int64_t>(T) * H * (kDv / 8);   // in 16-byte vectors
  const uint4* src = reinterpret_cast<const uint4*>(ws_o) + th * (kDv / 8) + 2 * lane;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int s0 = 0; s0 < n_split; s0 += kCombineBatch) {
    const int nb = min(kCombineBatch, n_split - s0);
    uint4 v[kCombineBatch][2];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (u < nb) {
        v[u][0] = __ldcs(src + (s0 + u) * slice_stride);
        v[u][1] = __ldcs(src + (s0 + u) * slice_stride + 1);
      }
    }
    const float ls = lane < nb ? ws_lse[(static_cast<int64_t>(s0 + lane) * T + t) * H + h] : -INFINITY;
    float mb = ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float m_new = fmaxf(m, mb);
    // previous batches rescaled to the new maximum (all zero while m is -inf)
    const float f = (m == -INFINITY) ? 0.f : __expf(m - m_new);
    const float wl = (ls == -INFINITY) ? 0.f : __expf(ls - m_new);
    float wsum = wl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    l = l * f + wsum;
    m = m_new;
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] *= f;
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const float ww = __shfl_sync(0xffffffffu, wl, u);
      if (u < nb) {
        const uint32_t w8[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc[2 * k] = fmaf(ww, __uint_as_float(w8[k] << 16), acc[2 * k]);
          acc[2 * k + 1] = fmaf(ww, __uint_as_float(w8[k] & 0xFFFF0000u), acc[2 * k + 1]);
        }
      }
    }
  }
  if (lane == 0 && lse_out) lse_out[th] = l > 0.f ? m + logf(l) : -INFINITY;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  uint32_t pk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
  uint4* dst = reinterpret_cast<uint4*>(out + th * kDv) + 2 * lane;
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

bool tc_supported(const SeqArgs& seq, const MlaArgs& a) {
  if (a.H != kH || a.d_latent != kDv || a.d_rope != kDqk - kDv) return false;
  if (a.kind == MlaKind::kF32) return false;
  if (a.kind == MlaKind::kBF16 && a.row_bytes % 16 != 0) return false;
  if (a.kind == MlaKind::kFP8Row && a.row_bytes % 16 != 0) return false;
  if (reinterpret_cast<uintptr_t>(a.kv) % 16 || reinterpret_cast<uintptr_t>(a.q) % 16 ||
      reinterpret_cast<uintptr_t>(a.out) % 16)
    return false;
  (void)seq;
  return true;
}

// Row slices per query: fill the GPU with (query, half, slice) CTAs, at least
// 4 tiles (128 rows) per slice, at most 64 slices.
int choose_split(const SeqArgs& seq, const MlaArgs& a, int num_sms) {
  const int max_split = std::min(64, std::max(1, (a.K + 4 * kBR - 1) / (4 * kBR)));
  const int64_t ctas = 2ll * seq.T;
  int split = 1;
  while (split < max_split && ctas * split * 2 <= num_sms) split *= 2;
  return std::min(split, max_split);
}

}  // namespace

size_t attn_workspace_bytes(const SeqArgs& seq, const MlaArgs& a, int num_sms) {
  if (!tc_supported(seq, a) || seq.T == 0) return 0;
  const int split = choose_split(seq, a, num_sms);
  if (split <= 1) return 0;
  const size_t o = static_cast<size_t>(split) * seq.T * kH * kDv * sizeof(uint16_t);
  const size_t l = static_cast<size_t>(split) * seq.T * kH * sizeof(float);
  return ((o + 255) / 256) * 256 + ((l + 255) / 256) * 256;
}

cudaError_t launch_attn(const SeqArgs& seq, const MlaArgs& a, void* workspace, size_t ws_bytes,
                        const LaunchEnv& env, std::string* plan, bool* unsupported,
                        std::string* why) {
  *unsupported = false;
  if (seq.T == 0) {
    *plan += "attn[empty]";
    return cudaSuccess;
  }
  if (tc_supported(seq, a)) {
    const bool fp8 = a.kind == MlaKind::kFP8Row;
    const int tile_rows = fp8 ? kBR : kBR48;
    int split = choose_split(seq, a, env.num_sms);
    if (split > 1 && (workspace == nullptr || ws_bytes < attn_workspace_bytes(seq, a, env.num_sms)))
      split = 1;  // no room for partials: one slice per query
    const int rps = ((a.K + split - 1) / split + tile_rows - 1) / tile_rows * tile_rows;
    split = (a.K + rps - 1) / rps;  // every slice non-empty
    TcAttnParams p{seq, a, split, rps, nullptr, nullptr};
    if (split > 1) {
      const size_t o = static_cast<size_t>(split) * seq.T * kH * kDv * sizeof(uint16_t);
      p.ws_o = static_cast<uint16_t*>(workspace);
      p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o + 255) / 256) * 256);
    }
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
      attr_err = cudaFuncSetAttribute(attn_tc48_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kT48SmemBytes);
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        AttnCfg<true>::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int grid = seq.T * split * 2;
    if (fp8) {
      const cudaError_t le =
          launch_kernel(attn_tc_kernel<true>, dim3(grid), dim3(kThreads), AttnCfg<true>::kSmemBytes, env.stream, true, 1, p);
      if (le != cudaSuccess) return le;
    } else {
      const cudaError_t le =
          launch_kernel(attn_tc48_kernel, dim3(grid), dim3(kT48Threads), kT48SmemBytes, env.stream, true, 1, p);
      if (le != cudaSuccess) return le;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    char buf[128];
    snprintf(buf, sizeof(buf), "attn_tc<%s>[split=%d,grid=%d]", fp8 ? "fp8" : "bf16x48", split, grid);
    *plan += buf;
    if (split > 1) {
      e = launch_kernel(attn_combine_kernel, dim3(seq.T, kH / kCombineHeads), dim3(32 * kCombineHeads), 0, env.stream,
                        true, 1,
                     static_cast<const uint16_t*>(p.ws_o), static_cast<const float*>(p.ws_lse), split, seq.T,
                     static_cast<__nv_bfloat16*>(a.out), a.lse);
      if (e != cudaSuccess) return e;
      *plan += "+attn_combine";
      e = cudaGetLastError();
    }
    return e;
  }
  const int dqk = a.d_latent + a.d_rope;
  const size_t smem = static_cast<size_t>(dqk) * 4 + static_cast<size_t>(a.K) * 8;
  if (smem > 200 * 1024) {
    *unsupported = true;
    *why = "attn: K or head dim too large for the generic kernel";
    return cudaSuccess;
  }
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(attn_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
  dim3 grid(a.H, seq.T);
  const cudaError_t le = launch_kernel(attn_generic_kernel, grid, dim3(kGenThreads), smem, env.stream, true, 1, seq, a);
  if (le != cudaSuccess) return le;
  *plan += "attn_generic";
  return cudaGetLastError();
}

}  // namespace dsa
