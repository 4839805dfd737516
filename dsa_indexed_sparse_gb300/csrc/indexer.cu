// Lightning-indexer scores (step 1 of the DSA path).
//
// "Day0 Inference Adaptation and Performance Optimization for Kimi K3.1 Pro",
// section 3: relevance scores between each query and every historical position,
// weighted by per-head weights, read from the paged key cache.  Per query t and
// causal position s <= q_pos[t]:
//     I[t, s] = sum_h w[t,h] * ReLU(q_I[t,h] . k_I[s])
// with q_I = q_code * q_scale[t,h] and k_I = k_code * k_scale[s].  Because the
// scales are positive, the kernels factor them out of the ReLU:
//     I[t, s] = k_scale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(q_code . k_code)
//
// Two kernels:
//  * indexer_tc_kernel<G> -- the tensor-core path (FP8 e4m3, H_I = 64, D_I = 128,
//    64-token pages).  Swap-AB tcgen05 GEMM: the 128 keys of a tile are the M
//    rows (TMEM lanes), the G queries x 64 heads of a query group are the N
//    columns, K = 128.  Keys arrive page by page through TMA (128-byte swizzle)
//    and their per-key scales through one warp-wide cp.async per tile (a TMA op
//    costs ~0.1 us of issue time on this GPU, which paced the whole ring when
//    the scales took two more); accumulators live in TMEM (double buffered) and
//    4*G epilogue warps, one per (query, TMEM lane quarter), turn each key's 64
//    dot products of a query into its score with an in-thread head sum.
//    Persistent: every CTA takes an equal contiguous share of the (group, key
//    tile) list, computed on the device from q_pos.
//  * indexer_generic_kernel -- CUDA cores, any H_I/D_I, fp32 or e4m3.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"
#include "topk_select.cuh"

DSA_DEFINE_STATUS_WORD(indexer)

namespace dsa {
namespace {

// =============================================================== generic kernel
constexpr int kGenThreads = 256;

// kFmt: 0 fp32 values, 1 e4m3 codes with fp32 per-token / per-head scales,
// 2 MXFP8 (e4m3 codes, E8M0 scale per 32 elements: the query is dequantised
// into shared memory and each key element is dequantised as it is read; both
// are exact in fp32).
template <int kFmt>
__global__ void __launch_bounds__(kGenThreads)
    indexer_generic_kernel(SeqArgs seq, IndexerArgs a) {
  grid_dep_wait();
  extern __shared__ float sm_gen[];
  float* qf = sm_gen;                   // [H_I * D_I] query values (codes for kFmt 1)
  float* wq = sm_gen + a.H_I * a.D_I;  // [H_I] w * q_scale (w for MXFP8)
  const int t = blockIdx.y;
  const int qpos = __ldg(seq.q_pos + t);
  const int b = __ldg(seq.q_seq + t);
  if (qpos < 0 || qpos >= seq.max_ctx || b < 0 || b >= seq.B) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(&g_status_indexer, kDevBadPos);
    return;
  }
  const int HD = a.H_I * a.D_I;
  const int nb = a.D_I / 32;            // MXFP8 blocks per vector
  for (int i = threadIdx.x; i < HD; i += blockDim.x) {
    if (kFmt == 0) {
      qf[i] = static_cast<const float*>(a.q)[static_cast<int64_t>(t) * HD + i];
    } else {
      float v = e4m3_to_float(static_cast<const uint8_t*>(a.q)[static_cast<int64_t>(t) * HD + i]);
      if (kFmt == 2) {
        const int h = i / a.D_I, blk = (i % a.D_I) / 32;
        const int e = static_cast<const uint8_t*>(a.q_scale)[(static_cast<int64_t>(t) * a.H_I + h) * nb + blk];
        v = ldexpf(v, e - 127);
      }
      qf[i] = v;
    }
  }
  for (int h = threadIdx.x; h < a.H_I; h += blockDim.x) {
    const float sq = (kFmt != 2 && a.q_scale)
                         ? __ldg(static_cast<const float*>(a.q_scale) + static_cast<int64_t>(t) * a.H_I + h)
                         : 1.f;
    wq[h] = __ldg(a.w + static_cast<int64_t>(t) * a.H_I + h) * sq;
  }
  __syncthreads();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s > qpos) return;
  const int64_t row = phys_row(seq.block_table + static_cast<int64_t>(b) * seq.bt_stride, s,
                               seq.page_size, seq.n_pages, &g_status_indexer);
  if (row < 0) return;
  float acc = 0.f;
  for (int h = 0; h < a.H_I; ++h) {
    float d = 0.f;
    if (kFmt == 0) {
      const float* kr = static_cast<const float*>(a.k) + row * a.D_I;
      for (int i = 0; i < a.D_I; ++i) d = fmaf(qf[h * a.D_I + i], kr[i], d);
    } else if (kFmt == 1) {
      const uint8_t* kr = static_cast<const uint8_t*>(a.k) + row * a.D_I;
      for (int i = 0; i < a.D_I; ++i) d = fmaf(qf[h * a.D_I + i], e4m3_to_float(kr[i]), d);
    } else {
      const uint8_t* kr = static_cast<const uint8_t*>(a.k) + row * a.D_I;
      const uint8_t* ke = static_cast<const uint8_t*>(a.k_scale) + row * nb;
      for (int i = 0; i < a.D_I; ++i)
        d = fmaf(qf[h * a.D_I + i], ldexpf(e4m3_to_float(kr[i]), static_cast<int>(ke[i / 32]) - 127), d);
    }
    acc = fmaf(wq[h], fmaxf(d, 0.f), acc);
  }
  const float sk = (kFmt != 2 && a.k_scale) ? __ldg(static_cast<const float*>(a.k_scale) + row) : 1.f;
  a.scores[static_cast<int64_t>(t) * a.ld + s] = acc * sk;
}

// =============================================================== tcgen05 kernel
constexpr int kTcHeads = 64;       // H_I
constexpr int kTcDim = 128;        // D_I (bytes per key row)
constexpr int kTcKeys = 128;       // keys per tile = UMMA M
constexpr int kTcPage = 64;        // tokens per page
constexpr int kTcStages = 6;       // key-tile ring depth (16 KB each)
// Waiting warps sleep between polls (woken when the phase completes): spinning
// epilogue warps took the issue slots of the TMA producer on their sub-partition
// (one tile issued every ~0.45 us).
constexpr uint32_t kSleepNs = 1000;
// warp 0 TMA, warp 1 MMA, then the epilogue: one warp per (query of the group,
// TMEM lane quarter) in each of kRot groups that take the tiles in turn (tile it
// goes to group it % kRot), so 4*G*kRot warps.  The ReLU-weighted head sums (two
// CUDA-core operations per key, query and head) cost about as much issue time as
// the MMAs' tensor time at prefill, so they get every warp slot the register
// budget allows; with one query per group, four groups rotating over the tiles
// keep one tile's head sums from pacing the key stream.  (Splitting a single
// query's heads over two warps per quarter made the decode configurations
// slower.)
// Every per-tile role is a chain of dependent issue steps that takes one warp
// ~0.4 us a tile (the copies: page lookup, barrier arrival, TMA, the scales'
// cp.async; the MMAs: barrier waits, descriptors, four MMAs, two commits), which
// capped an SM at ~37 GB/s of keys: kProd producer warps and kMmaWarps issuing
// warps take the tiles in turn as the epilogue groups do.
template <int G, bool kMx = false>
struct TcWarps {
  static constexpr int kRot = G == 1 ? (kMx ? 2 : 3) : 1;
  static constexpr int kProd = 2;                  // divides kTcStages
  static constexpr int kMmaWarps = G == 1 ? 2 : 1;
  static constexpr int kMma = kProd;               // the first MMA-issuing warp (also allocates TMEM)
  static constexpr int kEpi0 = kProd + kMmaWarps;  // first epilogue warp
  static constexpr int kEpiWarps = 4 * G * kRot;
  static constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
};

// kMx: MXFP8 keys and queries (E8M0 scale per 32 elements).  The four 32-wide
// blocks of the K = 128 dot product go to four separate accumulators (one
// MMA each, no accumulation), which the epilogue scales by the two blocks'
// power-of-two factors and sums: d = sum_b 2^(eq_b + ek_b - 254) * D_b.
template <int G, bool kMx = false>
struct TcCfg {
  static_assert(!kMx || G == 1, "MXFP8 keys run one query per group");
  static constexpr int N = kTcHeads * G;                 // UMMA N
  static constexpr int kBlocks = kMx ? kTcDim / 32 : 1;  // accumulators per tile
  static constexpr int kAccCols = kBlocks * N;           // TMEM columns per tile
  static constexpr int kStageBytes = kTcKeys * kTcDim;   // 16384
  static constexpr int kQBytes = N * kTcDim;             // one query-group buffer
  // accumulator buffers: two, or one per rotation group
  static constexpr int kAccBufs = TcWarps<G, kMx>::kRot > 2 ? TcWarps<G, kMx>::kRot : 2;
  static constexpr int kTmemNeed = kAccBufs * kAccCols;
  static_assert(kTmemNeed <= 512, "TMEM plan");
  static constexpr uint32_t kTmemCols = kTmemNeed <= 128 ? 128u : (kTmemNeed <= 256 ? 256u : 512u);
  // per epilogue warp: w / 2 for its 64 heads, then (MXFP8) the query's block
  // factors 2^(e - 127) as float [4][64]
  static constexpr int kSlice = kTcHeads * (1 + (kMx ? kBlocks : 0));
  static constexpr int kOffStages = 0;
  static constexpr int kOffQ = kOffStages + kTcStages * kStageBytes;
  static constexpr int kOffWq = kOffQ + 2 * kQBytes;      // float [4G][kSlice]: each epilogue warp's slice
  // key scales: 4 bytes per key (an fp32 scale, or MXFP8's four E8M0 bytes)
  static constexpr int kOffScale = kOffWq + TcWarps<G, kMx>::kEpiWarps * kSlice * 4;
  static constexpr int kOffValid = kOffScale + kTcStages * kTcKeys * 4;  // uint32 [stages]
  static constexpr int kOffBar = kOffValid + kTcStages * 4 + 8;
  // barriers: full[S], empty[S], qfull[2], qempty[2], accfull[A], accempty[A], drain
  static constexpr int kNumBars = 2 * kTcStages + 4 + 2 * kAccBufs + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort, sched[2], red[one per warp]
  static constexpr int kSmemBytes = kOffMisc + 256 + 1024;  // + alignment slack
  // fused decode plan: the selection's scratch, then this CTA's keys (read 16
  // bytes at a time), both 128-byte aligned
  static constexpr int kOffSel = (kOffMisc + 256 + 127) / 128 * 128;
  static constexpr int kOffKeys = (kOffSel + static_cast<int>(sizeof(SelectSmem)) + 127) / 128 * 128;
  static_assert(kOffKeys % 16 == 0 && kOffSel % 16 == 0, "aligned fused-plan regions");
  static constexpr uint32_t kIdesc = make_idesc(kFmtE4M3, kFmtE4M3, false, false, kTcKeys, N);
};

// Keys of one query a CTA of the fused plan holds in shared memory at most.
constexpr int kFusedMaxKeys = 16384;
// Largest cluster (CTAs per query) the fused plan is chosen for.
constexpr int kFusedMaxCluster = 2;

struct TcParams {
  SeqArgs seq;
  IndexerArgs a;
  int32_t n_groups;
  // fused decode plan: the selection's K and the index rows [T, K]
  int32_t K;
  int32_t* idx;
};

// Number of 128-key tiles of query group g (its longest causal history), with
// q_pos validation.  Also returns the group's history length.
template <int G>
__device__ __forceinline__ int group_tiles(const TcParams& p, int g, int* n_hist) {
  int n = 0;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const int t = g * G + j;
    if (t < p.seq.T) {
      const int qp = __ldg(p.seq.q_pos + t);
      if (qp < 0 || qp >= p.seq.max_ctx) {
        atomicOr(&g_status_indexer, kDevBadPos);
      } else {
        n = max(n, qp + 1);
      }
    }
  }
  *n_hist = n;
  return (n + kTcKeys - 1) / kTcKeys;
}

// Walks the (group, key tile) list from a starting point.
template <int G>
struct TileWalker {
  int g, kt, ntiles, nhist;
  __device__ void init(const TcParams& p, int g0, int kt0) {
    g = g0;
    kt = kt0;
    ntiles = group_tiles<G>(p, g, &nhist);
  }
  __device__ void advance(const TcParams& p) {
    ++kt;
    while (kt >= ntiles && g + 1 < p.n_groups) {
      ++g;
      kt = 0;
      ntiles = group_tiles<G>(p, g, &nhist);
    }
  }
};

template <int kThreads>
__device__ __forceinline__ int block_sum(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
  return tot;
}

// kFused (one query per group): the fused decode plan.  A cluster of CTAs per
// query, each CTA streaming a contiguous run of its key tiles; the epilogue
// writes each score as an order key into this CTA's shared memory (never to
// global memory) and counts it into the first histogram; once the cluster's
// keys are complete the CTAs select the Top-K together and only the index row
// leaves the SM.
template <int G, bool kMx, bool kFused>
__global__ void __launch_bounds__(TcWarps<G, kMx>::kThreads, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap kmap2,
                      const __grid_constant__ CUtensorMap qmap, TcParams p) {
  static_assert(!kFused || G == 1, "the fused plan runs one query per group");
  using C = TcCfg<G, kMx>;
  constexpr int kTcThreads = TcWarps<G, kMx>::kThreads;
  constexpr int kRot = TcWarps<G, kMx>::kRot;
  constexpr int kProd = TcWarps<G, kMx>::kProd;
  constexpr int kMmaWarp = TcWarps<G, kMx>::kMma;
  constexpr int kMmaWarps = TcWarps<G, kMx>::kMmaWarps;
  constexpr int kEpi0 = TcWarps<G, kMx>::kEpi0;
  static_assert(kTcStages % kProd == 0, "each producer owns every kProd-th stage");
  constexpr int kGroupWarps = 4 * G;           // epilogue warps that share one tile
  constexpr int NB = C::kAccBufs;
  static_assert(4 + kTcThreads / 32 <= 64, "misc area holds one int per warp");
  // No grid_dep_wait() yet: the work split, barriers and TMEM (inputs only)
  // overlap the tail of the kernel before when that one lets this grid start early.
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // re-aligned by pointer arithmetic on the shared array, so that the compiler
  // keeps every access through `sm` in the shared window
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kTcStages;
  uint64_t* qfull = bars + 2 * kTcStages;
  uint64_t* qempty = qfull + 2;
  uint64_t* accfull = qfull + 4;
  uint64_t* accempty = accfull + NB;
  uint64_t* drain = accempty + NB;   // every MMA of the issuing warp complete (teardown)
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  int* sched = reinterpret_cast<int*>(misc + 2);   // g0, kt0
  int* red = reinterpret_cast<int*>(misc + 4);     // one int per warp
  float* wq_s = reinterpret_cast<float*>(sm + C::kOffWq);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  SelectSmem* sel = reinterpret_cast<SelectSmem*>(sm + C::kOffSel);
  uint32_t* keys_s = reinterpret_cast<uint32_t*>(sm + C::kOffKeys);
  int f_lo = 0, f_len = 0, f_CL = 1;   // fused: this CTA's slice of the query's history
  int32_t* f_out = nullptr;
  int64_t begin = 0, end = 0;
  if constexpr (kFused) {
    // ---- one query per cluster; an equal share of its tiles per CTA -----------
    f_CL = static_cast<int>(cl_size());
    const int rank = static_cast<int>(cl_rank());
    const int t = p.seq.T - 1 - static_cast<int>(blockIdx.x) / f_CL;
    int qp = __ldg(p.seq.q_pos + t);
    if (qp < 0 || qp >= p.seq.max_ctx) {
      if (threadIdx.x == 0 && rank == 0) atomicOr(&g_status_indexer, kDevBadPos);
      qp = -1;
    }
    const int n = qp + 1;
    f_out = p.idx + static_cast<int64_t>(t) * p.K;
    if (n <= p.K) {   // cluster-uniform: every position is kept, no score needed
      grid_dep_wait();   // the index row may still be read by the kernel before
      for (int i = rank * kTcThreads + threadIdx.x; i < p.K; i += f_CL * kTcThreads) f_out[i] = i < n ? i : -1;
      grid_dep_launch();
      return;
    }
    const int tiles = (n + kTcKeys - 1) / kTcKeys;
    const int kt0 = static_cast<int>(static_cast<int64_t>(rank) * tiles / f_CL);
    const int kt1 = static_cast<int>(static_cast<int64_t>(rank + 1) * tiles / f_CL);
    if (threadIdx.x == 0) {
      sched[0] = t;
      sched[1] = kt0;
    }
    begin = 0;
    end = kt1 - kt0;
    f_lo = kt0 * kTcKeys;
    f_len = max(0, min(n, kt1 * kTcKeys) - f_lo);
    select_prepare<kTcThreads>(sel, f_CL);   // zeroes the histograms, arrives at the cluster barrier
  } else {
  // ---- work split: equal share of the global tile list -----------------
  int total = 0;
  for (int g0 = 0; g0 < p.n_groups; g0 += kTcThreads) {
    const int g = g0 + threadIdx.x;
    int nh;
    const int c = (g < p.n_groups) ? group_tiles<G>(p, g, &nh) : 0;
    total += block_sum<kTcThreads>(c, red);
  }
  begin = static_cast<int64_t>(blockIdx.x) * total / gridDim.x;
  end = static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x;
  if (begin >= end) return;  // block-uniform
  {
    int run = 0;
    for (int g0 = 0; g0 < p.n_groups; g0 += kTcThreads) {
      const int g = g0 + threadIdx.x;
      int nh;
      const int c = (g < p.n_groups) ? group_tiles<G>(p, g, &nh) : 0;
      // inclusive scan within the block
      int v = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      __syncthreads();
      if (lane == 31) red[warp] = v;
      __syncthreads();
      int before = 0, chunk = 0;
      for (int w = 0; w < kTcThreads / 32; ++w) {
        if (w < warp) before += red[w];
        chunk += red[w];
      }
      const int excl = run + before + v - c;
      if (c > 0 && begin >= excl && begin < excl + c) {
        sched[0] = g;
        sched[1] = static_cast<int>(begin - excl);
      }
      run += chunk;
    }
  }
  }

  // ---- barriers and TMEM -------------------------------------------------
  if (threadIdx.x == 0) {
    // full: the producer's expect_tx arrival, plus one cp.async arrival per lane
    // of the producer warp when the keys carry scales (always for MXFP8)
    const uint32_t full_count = 1u + (p.a.k_scale != nullptr ? 32u : 0u);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], full_count);
      // freed by the MMA (keys read) and by each epilogue warp of the tile's
      // group (key scales read)
      mbar_init(&empty[i], 1 + kGroupWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kMmaWarps);   // each issuing warp releases a group's Q
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], kGroupWarps);
    }
    mbar_init(drain, kMmaWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&kmap2);
    tma_prefetch_desc(&qmap);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(misc, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int g_start = sched[0], kt_start = sched[1];
  const int ntiles = static_cast<int>(end - begin);   // <= total, an int
  // Producer pw's first own tile (it = pw): its group's sequence and page count
  // and the page ids of its first window, read before the wait -- step
  // metadata that no kernel of this library writes -- so that the first copies
  // go out right after it instead of after three dependent loads.  Only in CTAs
  // with more than two tiles: with one or two (decode batch 1) the CTAs that
  // start late, behind the kernels before, pay the longer set-up on the step's
  // critical path (A/B: decode b1 +0.17 us with it, long decode -0.65 us).
  int pre_g = -1, pre_kt = -1, pre_b = 0, pre_npg = 0;
  int32_t pre_page = -1;
  if (warp < kProd && ntiles > 2) {
    TileWalker<G> w0;
    w0.init(p, g_start, kt_start);
    for (int i = 0; i < warp; ++i) w0.advance(p);
    pre_g = w0.g;
    pre_kt = w0.kt;
    pre_b = __ldg(p.seq.q_seq + w0.g * G);
    pre_npg = (w0.nhist + kTcPage - 1) / kTcPage;
    const int lp = 2 * (pre_kt + (lane >> 1) * kProd) + (lane & 1);
    if (pre_b >= 0 && pre_b < p.seq.B && lp < pre_npg)
      pre_page = __ldg(p.seq.block_table + static_cast<int64_t>(pre_b) * p.seq.bt_stride + lp);
  }
  grid_dep_wait();

  if (warp < kProd) {
    // ------------------------------------------------ TMA producers (warps 0 .. kProd - 1)
    // Producer pw issues the copies of the tiles it with it % kProd == pw (and so
    // of the stages st with st % kProd == pw).  It keeps the page ids of its next
    // 16 tiles in registers (lane l: tile l / 2, page l % 2, loaded in parallel);
    // lane 0 issues the TMA tile loads, every lane one 16-byte copy of key
    // scales.  A query group's own TMA load goes with the producer of the
    // group's first tile in this CTA.
    const int pw = warp;
    TileWalker<G> w;
    w.init(p, g_start, kt_start);
    int cur_g = -1, qcount = 0;
    int win_kt = -1;        // kt of the window's first tile; the window holds kt, kt + kProd, ...
    int32_t my_page = -1;   // page id of window tile lane / 2, page lane % 2
    const int32_t* bt = p.seq.block_table;
    bool b_ok = false;
    int npg = 0;
    uint32_t* valid_s = reinterpret_cast<uint32_t*>(sm + C::kOffValid);
    float* scale_s = reinterpret_cast<float*>(sm + C::kOffScale);
    int issued = 0, last_it = -1;   // tiles whose copies this warp issued, the last of them
    uint32_t q_mine = 0;   // bit b: the last Q load into buffer b was issued by this warp
    for (int it = 0; it < ntiles; ++it, w.advance(p)) {
      if (w.g != cur_g) {
        const int qb = qcount & 1;
        const bool mine = it % kProd == pw;
        if (mine) {
          if (qcount >= 2) {
            const bool ok = mbar_wait(&qempty[qb], ((qcount >> 1) - 1) & 1, &g_status_indexer, abort_flag,
                                      kWaitLimitNs, kSleepNs);
            if (!__all_sync(0xffffffffu, ok)) break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&qfull[qb], C::kQBytes);
            tma_load_2d(sm + C::kOffQ + qb * C::kQBytes, &qmap, &qfull[qb], 0, w.g * G * kTcHeads);
          }
        }
        q_mine = mine ? (q_mine | (1u << qb)) : (q_mine & ~(1u << qb));
        const int b = w.g == pre_g ? pre_b : __ldg(p.seq.q_seq + w.g * G);
        b_ok = (b >= 0 && b < p.seq.B);
        bt = p.seq.block_table + static_cast<int64_t>(b_ok ? b : 0) * p.seq.bt_stride;
        npg = (w.nhist + kTcPage - 1) / kTcPage;
        win_kt = -1;
        cur_g = w.g;
        ++qcount;
      }
      if (it % kProd != pw) continue;
      if (win_kt < 0 || (w.kt - win_kt) / kProd >= 16) {
        const bool pre = w.g == pre_g && w.kt == pre_kt;   // the window read before the wait
        pre_g = -1;
        win_kt = w.kt;
        const int lp = 2 * (win_kt + (lane >> 1) * kProd) + (lane & 1);
        my_page = (b_ok && lp < npg) ? (pre ? pre_page : __ldg(bt + lp)) : -1;
        if (lp < npg && (my_page < 0 || my_page >= p.seq.n_pages || !b_ok)) {
          atomicOr(&g_status_indexer, kDevBadIndex);
          my_page = -1;
        }
      }
      const int wi = 2 * ((w.kt - win_kt) / kProd);
      const int32_t pid0 = __shfl_sync(0xffffffffu, my_page, wi);
      int32_t pid1 = __shfl_sync(0xffffffffu, my_page, wi + 1);
      if (2 * w.kt + 1 >= npg) pid1 = -1;
      const int st = it % kTcStages;
      if (it >= kTcStages) {
        const bool ok = mbar_wait(&empty[st], ((it / kTcStages) - 1) & 1, &g_status_indexer, abort_flag,
                                  kWaitLimitNs, kSleepNs);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) {
        constexpr uint32_t per_page = C::kStageBytes / 2;
        valid_s[st] = (pid0 >= 0 ? 1u : 0u) | (pid1 >= 0 ? 2u : 0u);
        mbar_arrive_expect_tx(&full[st], (pid0 >= 0 ? per_page : 0u) + (pid1 >= 0 ? per_page : 0u));
        uint8_t* dst = sm + C::kOffStages + st * C::kStageBytes;
        // two adjacent pages go in one 128-row box (kmap2), the others one page each
        if (pid0 >= 0 && pid1 == pid0 + 1) {
          tma_load_2d(dst, &kmap2, &full[st], 0, pid0 * kTcPage);
        } else {
          if (pid0 >= 0) tma_load_2d(dst, &kmap, &full[st], 0, pid0 * kTcPage);
          if (pid1 >= 0) tma_load_2d(dst + C::kStageBytes / 2, &kmap, &full[st], 0, pid1 * kTcPage);
        }
      }
      if (p.a.k_scale != nullptr) {
        // lanes 0-15: the 64 scales of the first page, lanes 16-31: the second (16 B each)
        const int half = lane >> 4;
        const int32_t pid = half ? pid1 : pid0;
        if (pid >= 0)
          cp_async16(smem_u32(scale_s + st * kTcKeys + half * kTcPage + (lane & 15) * 4),
                     static_cast<const uint8_t*>(p.a.k_scale) +
                         (static_cast<int64_t>(pid) * kTcPage + (lane & 15) * 4) * 4);
        cp_async_mbar_arrive(&full[st]);
      }
      ++issued;
      last_it = it;
    }
    // On the way out (also after an abort) every copy this warp issued has landed
    // before the CTA's shared memory is released: its last tiles, one per stage
    // it owns, and the Q loads of the last two groups if it issued them, each in
    // the phase of its last use.
    for (int m = 0; m < min(issued, kTcStages / kProd); ++m) {
      const int k = last_it - m * kProd;
      mbar_drain(&full[k % kTcStages], (k / kTcStages) & 1, &g_status_indexer);
    }
    for (int k = max(0, qcount - 2); k < qcount; ++k)
      if ((q_mine >> (k & 1)) & 1u) mbar_drain(&qfull[k & 1], (k >> 1) & 1, &g_status_indexer);
  } else if (warp < kMmaWarp + kMmaWarps) {
    // ------------------------------------------------ MMA issuers (whole warps, an elected lane issues)
    // Issuing warp mw takes the tiles it with it % kMmaWarps == mw.  Every issuing
    // warp waits for each group's Q and releases it (its commit arrives once its
    // own MMAs on it are done), so no warp can release a buffer's next group
    // before that group's Q has landed.
    const int mw = warp - kMmaWarp;
    TileWalker<G> w;
    w.init(p, g_start, kt_start);
    int cur_g = -1, qcount = 0, qb = 0;
    for (int it = 0; it < ntiles; ++it, w.advance(p)) {
      if (w.g != cur_g) {
        if (qcount > 0) {
          if (elect_one()) umma_commit(&qempty[qb]);  // previous group's MMAs release its Q
          __syncwarp();
        }
        qb = qcount & 1;
        const bool ok = mbar_wait(&qfull[qb], (qcount >> 1) & 1, &g_status_indexer, abort_flag, kWaitLimitNs, kSleepNs);
        if (!__all_sync(0xffffffffu, ok)) break;
        cur_g = w.g;
        ++qcount;
      }
      if (kMmaWarps > 1 && it % kMmaWarps != mw) continue;
      const int st = it % kTcStages;
      bool ok = mbar_wait(&full[st], (it / kTcStages) & 1, &g_status_indexer, abort_flag, kWaitLimitNs, kSleepNs);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int ab = it % NB;
      if (it >= NB) {
        ok = mbar_wait(&accempty[ab], ((it / NB) - 1) & 1, &g_status_indexer, abort_flag, kWaitLimitNs, kSleepNs);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      tc_fence_after();
      // descriptors built once per tile; the unrolled K loop adds 32-byte steps to
      // the start-address field; one elected lane issues the block
      const uint64_t da = make_sdesc(smem_u32(sm + C::kOffStages + st * C::kStageBytes), 16, 1024, kLayoutSw128);
      const uint64_t db = make_sdesc(smem_u32(sm + C::kOffQ + qb * C::kQBytes), 16, 1024, kLayoutSw128);
      const uint32_t dcol = tmem + ab * C::kAccCols;
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < kTcDim / 32; ++k) {
          if (kMx)   // block k into its own accumulator
            umma_f8(dcol + k * C::N, da + static_cast<uint64_t>(2 * k), db + static_cast<uint64_t>(2 * k), C::kIdesc, 0u);
          else
            umma_f8(dcol, da + static_cast<uint64_t>(2 * k), db + static_cast<uint64_t>(2 * k), C::kIdesc,
                    k > 0 ? 1u : 0u);
        }
        umma_commit(&empty[st]);
        umma_commit(&accfull[ab]);
      }
      __syncwarp();
    }
    // every MMA this warp issued has finished before TMEM is released
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    mbar_drain(drain, 0, &g_status_indexer);
  } else {
    // ------------------------------------------------ epilogue (warps kEpi0 ..)
    // Warp e reduces query j = e / 4 of every group over the 32 keys of TMEM lane
    // quarter warp % 4.  Its head weights (w * q_scale) live in its own 64-float
    // slice of shared memory; the next group's weights and positions are fetched
    // into registers while the current group runs, so a group switch costs no
    // global-memory round trip.
    const int e = warp - kEpi0;
    const int quarter = warp & 3;   // the TMEM lanes a warp may read: 32 * (warp % 4) ..
    const int rg = e / kGroupWarps;           // rotation group: tiles it with it % kRot == rg
    const int j = (e % kGroupWarps) >> 2;     // query of the group
    const int row = quarter * 32 + lane;          // key within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float* wq = wq_s + e * C::kSlice;
    float* cq = wq + kTcHeads;   // MXFP8: the query's block factors [4][64]
    TileWalker<G> w;
    w.init(p, g_start, kt_start);
    int cur_g = -1, qp = -1;
    float* srow = p.a.scores;   // this warp's query's score row
    const uint32_t valid_addr = smem_u32(sm + C::kOffValid);
    const uint32_t scale_addr = smem_u32(sm + C::kOffScale) + row * 4;
    // prefetched group: its first query's sequence, this warp's query's sequence
    // and position, and lanes' two head weights and query scales
    int pf_g = -1, pf_b = 0, pf_qs = 0, pf_qp = -1;
    float pf_w0 = 0.f, pf_w1 = 0.f, pf_s0 = 1.f, pf_s1 = 1.f;
    uint32_t pf_e0 = 0x7F7F7F7Fu, pf_e1 = 0x7F7F7F7Fu;   // MXFP8: the two heads' four E8M0 bytes
    auto prefetch = [&](int g) {
      pf_g = g;
      const int t = g * G + j;
      pf_b = __ldg(p.seq.q_seq + g * G);
      pf_qs = pf_b;
      pf_qp = -1;
      pf_w0 = pf_w1 = 0.f;
      pf_s0 = pf_s1 = 1.f;
      if (t < p.seq.T) {
        pf_qs = __ldg(p.seq.q_seq + t);
        pf_qp = __ldg(p.seq.q_pos + t);
        const int64_t o = static_cast<int64_t>(t) * kTcHeads + 2 * lane;
        pf_w0 = __ldg(p.a.w + o);
        pf_w1 = __ldg(p.a.w + o + 1);
        if (kMx) {
          pf_e0 = __ldg(static_cast<const uint32_t*>(p.a.q_scale) + o);
          pf_e1 = __ldg(static_cast<const uint32_t*>(p.a.q_scale) + o + 1);
        } else if (p.a.q_scale) {
          pf_s0 = __ldg(static_cast<const float*>(p.a.q_scale) + o);
          pf_s1 = __ldg(static_cast<const float*>(p.a.q_scale) + o + 1);
        }
      }
    };
    for (int it = 0; it < ntiles; ++it, w.advance(p)) {
      if (kRot > 1 && it % kRot != rg) continue;
      if (w.g != cur_g) {
        if (pf_g != w.g) prefetch(w.g);
        const int tq = w.g * G + j;
        qp = (tq < p.seq.T && pf_qp < p.seq.max_ctx) ? pf_qp : -1;
        srow = p.a.scores + static_cast<int64_t>(tq < p.seq.T ? tq : 0) * p.a.ld;
        if (tq < p.seq.T && pf_qs != pf_b && lane == 0) atomicOr(&g_status_indexer, kDevBadGroup);
        if (pf_b < 0 || pf_b >= p.seq.B) {
          if (lane == 0) atomicOr(&g_status_indexer, kDevBadIndex);
          qp = -1;
        }
        // the previous group's tiles are done: this warp alone reads its slice.
        // Half weights: w * ReLU(x) = (w / 2) * (x + |x|) exactly (the halving and
        // doubling are exact), and x + |x| runs on the FMA pipe instead of a
        // max on the half-rate ALU pipe.
        wq[2 * lane] = 0.5f * (pf_w0 * pf_s0);
        wq[2 * lane + 1] = 0.5f * (pf_w1 * pf_s1);
        if (kMx) {
#pragma unroll
          for (int bk = 0; bk < C::kBlocks; ++bk) {
            cq[bk * kTcHeads + 2 * lane] = ldexpf(1.f, static_cast<int>((pf_e0 >> (8 * bk)) & 0xFFu) - 127);
            cq[bk * kTcHeads + 2 * lane + 1] = ldexpf(1.f, static_cast<int>((pf_e1 >> (8 * bk)) & 0xFFu) - 127);
          }
        }
        __syncwarp();
        cur_g = w.g;
        if (w.g + 1 < p.n_groups) prefetch(w.g + 1);
      }
      const int ab = it % NB;
      bool ok = mbar_wait(&accfull[ab], (it / NB) & 1, &g_status_indexer, abort_flag, kWaitLimitNs, kSleepNs);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      // the stage (keys, scales, page validity) is still this tile's: the
      // producer refills it only after this warp's arrival on empty[st]
      const int st = it % kTcStages;
      ok = mbar_wait(&full[st], (it / kTcStages) & 1, &g_status_indexer, abort_flag, kWaitLimitNs, kSleepNs);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int s = w.kt * kTcKeys + row;
      uint32_t vmask;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(vmask) : "r"(valid_addr + st * 4) : "memory");
      const bool key_ok = s < w.nhist && ((vmask >> (row >> 6)) & 1u);
      float sk = 1.f;
      uint32_t ek = 0;   // MXFP8: this key's four E8M0 bytes
      if (kMx)
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(ek) : "r"(scale_addr + st * (kTcKeys * 4)) : "memory");
      else if (p.a.k_scale)
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sk) : "r"(scale_addr + st * (kTcKeys * 4)) : "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      const float4* w4 = reinterpret_cast<const float4*>(wq);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if constexpr (kMx) {
        // d[h] = sum_b D_b[h] * 2^(eq_b[h] - 127) * 2^(ek_b - 127), 32 heads at a time
        const uint32_t col = tmem + lane_off + ab * C::kAccCols;
        float kx[C::kBlocks];
#pragma unroll
        for (int bk = 0; bk < C::kBlocks; ++bk) kx[bk] = ldexpf(1.f, static_cast<int>((ek >> (8 * bk)) & 0xFFu) - 127);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float d[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) d[i] = 0.f;
#pragma unroll
          for (int bk = 0; bk < C::kBlocks; ++bk) {
            uint32_t v[32];
            tmem_ld32(col + bk * C::N + 32 * hh, v);
            tmem_ld_wait();
            if (hh == 1 && bk == C::kBlocks - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&accempty[ab]);   // the accumulators are in registers
            }
            // packed over head pairs: f = query factor * key factor, d += D * f
            const float4* c4 = reinterpret_cast<const float4*>(cq + bk * kTcHeads + 32 * hh);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 cv = c4[i];
              float f0, f1, f2, f3;
              mul2(f0, f1, cv.x, cv.y, kx[bk], kx[bk]);
              mul2(f2, f3, cv.z, cv.w, kx[bk], kx[bk]);
              fma2(d[4 * i], d[4 * i + 1], __uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), f0, f1);
              fma2(d[4 * i + 2], d[4 * i + 3], __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]), f2, f3);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 wv = w4[8 * hh + i];
            const int a = 4 * (i & 1);
            fma2(acc[a], acc[a + 1], wv.x, wv.y, d[4 * i] + fabsf(d[4 * i]), d[4 * i + 1] + fabsf(d[4 * i + 1]));
            fma2(acc[a + 2], acc[a + 3], wv.z, wv.w, d[4 * i + 2] + fabsf(d[4 * i + 2]),
                 d[4 * i + 3] + fabsf(d[4 * i + 3]));
          }
        }
      } else {
        // the 64 heads in two halves of 32 columns (fewer live registers: 18 warps
        // leave 96 a thread); head weights as 16-byte broadcast loads
        const uint32_t col = tmem + lane_off + ab * C::N + j * kTcHeads;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tmem_ld32(col + 32 * hh, v);
          tmem_ld_wait();
          if (hh == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[ab]);   // the accumulator is in registers
          }
          // x + |x| per head, then packed fmas over head pairs: eight running sums
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 wv = w4[8 * hh + i];
            const int a = 4 * (i & 1);
            float y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float x = __uint_as_float(v[4 * i + k]);
              y[k] = x + fabsf(x);
            }
            fma2(acc[a], acc[a + 1], wv.x, wv.y, y[0], y[1]);
            fma2(acc[a + 2], acc[a + 3], wv.z, wv.w, y[2], y[3]);
          }
        }
      }
      const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      if constexpr (kFused) {
        // a key on a bad page (flagged above) gets the lowest key of all
        if (s <= qp) {
          const uint32_t k = key_ok ? order_key(sum * sk) : 0u;
          keys_s[s - f_lo] = k;
          select_count0(sel, k);
        }
      } else {
        if (key_ok && s <= qp) srow[s] = sum * sk;
      }
    }
  }

  grid_dep_launch();  // this CTA's work is done: the next kernel may launch
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if constexpr (kFused) {
    // this CTA's keys are complete (the barrier above); select over the cluster
    select_run<kTcThreads>(
        sel, [&](int i) -> uint32_t { return keys_s[i]; },
        [&](int i) -> uint4 { return reinterpret_cast<const uint4*>(keys_s)[i >> 2]; }, f_len, f_lo, p.K, f_out,
        true);
  }
}

template <int G, bool kMx = false>
cudaError_t launch_tc(const SeqArgs& seq, const IndexerArgs& a, const LaunchEnv& env,
                      std::string* plan, bool* unsupported, std::string* why) {
  using C = TcCfg<G, kMx>;
  alignas(64) CUtensorMap kmap, kmap2, qmap;
  if (!encode_tmap_2d_u8(&kmap, a.k, kTcDim, static_cast<uint64_t>(seq.cache_rows), kTcDim,
                         kTcDim, kTcPage, why) ||
      !encode_tmap_2d_u8(&kmap2, a.k, kTcDim, static_cast<uint64_t>(seq.cache_rows), kTcDim,
                         kTcDim, 2 * kTcPage, why) ||
      !encode_tmap_2d_u8(&qmap, a.q, kTcDim, static_cast<uint64_t>(seq.T) * kTcHeads, kTcDim,
                         kTcDim, C::N, why)) {
    *unsupported = true;
    return cudaSuccess;
  }
  TcParams p{seq, a, (seq.T + G - 1) / G, 0, nullptr};
  const int64_t tiles_ub =
      static_cast<int64_t>(p.n_groups) * ((seq.max_ctx + kTcKeys - 1) / kTcKeys);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles_ub, env.num_sms)));
  const cudaError_t attr_err =
      ensure_smem_limit(reinterpret_cast<const void*>(indexer_tc_kernel<G, kMx, false>), C::kSmemBytes, env.device);
  if (attr_err != cudaSuccess) return attr_err;
  const cudaError_t le = launch_kernel(indexer_tc_kernel<G, kMx, false>, dim3(grid), dim3(TcWarps<G, kMx>::kThreads), C::kSmemBytes,
                                       env.stream, true, 1,
                                    kmap, kmap2, qmap, p);
  if (le != cudaSuccess) return le;
  char buf[160];
  snprintf(buf, sizeof(buf), "indexer_tc<G=%d%s>[grid=%d,tiles<=%lld]", G, kMx ? ",mxfp8" : "", grid,
           static_cast<long long>(tiles_ub));
  *plan += buf;
  return cudaGetLastError();
}

// Fused decode plan (indexer + Top-K, scores in shared memory): clusters of CL
// CTAs, one cluster per query.  CL: the whole GPU in one wave at small batch
// (up to 16 CTAs per query, non-portable cluster size), and enough CTAs that a
// slice's keys fit kFusedMaxKeys.  Returns CL, or 0 when the plan does not apply.
template <bool kMx>
int fused_cluster(const SeqArgs& seq, const LaunchEnv& env, int max_cl) {
  const int need = (seq.max_ctx + kFusedMaxKeys - 1) / kFusedMaxKeys;
  int cl = 1;
  while (cl < 16 && static_cast<int64_t>(seq.T) * cl * 2 <= env.num_sms) cl *= 2;
  cl = std::max(cl, need);
  if (cl > 16 || cl > max_cl) return 0;
  // every cluster of the launch resident at once is not required, but a cluster
  // of this size must fit on the GPU
  using C = TcCfg<1, kMx>;
  const int keys = (((seq.max_ctx + kTcKeys - 1) / kTcKeys + cl - 1) / cl) * kTcKeys;
  const size_t smem = static_cast<size_t>(C::kOffKeys) + static_cast<size_t>(keys) * 4 + 1024;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, TcParams) = indexer_tc_kernel<1, kMx, true>;
  if (ensure_smem_limit(reinterpret_cast<const void*>(kern),
                        C::kOffKeys + kFusedMaxKeys * 4 + 1024, env.device) != cudaSuccess)
    return 0;
  while (cl > 1 && !cluster_fits(reinterpret_cast<const void*>(kern), env.device, cl, TcWarps<1, kMx>::kThreads, smem)) {
    cl /= 2;
    if (cl < need) return 0;
  }
  return cl;
}

template <bool kMx>
cudaError_t launch_fused(const SeqArgs& seq, const IndexerArgs& a, int32_t K, int32_t* idx, int cl,
                         const LaunchEnv& env, std::string* plan, std::string* why, bool* unsupported) {
  using C = TcCfg<1, kMx>;
  alignas(64) CUtensorMap kmap, kmap2, qmap;
  if (!encode_tmap_2d_u8(&kmap, a.k, kTcDim, static_cast<uint64_t>(seq.cache_rows), kTcDim, kTcDim, kTcPage, why) ||
      !encode_tmap_2d_u8(&kmap2, a.k, kTcDim, static_cast<uint64_t>(seq.cache_rows), kTcDim, kTcDim, 2 * kTcPage,
                         why) ||
      !encode_tmap_2d_u8(&qmap, a.q, kTcDim, static_cast<uint64_t>(seq.T) * kTcHeads, kTcDim, kTcDim, C::N, why)) {
    *unsupported = true;
    return cudaSuccess;
  }
  TcParams p{seq, a, seq.T, K, idx};
  const int keys = (((seq.max_ctx + kTcKeys - 1) / kTcKeys + cl - 1) / cl) * kTcKeys;
  const size_t smem = static_cast<size_t>(C::kOffKeys) + static_cast<size_t>(keys) * 4 + 1024;
  const cudaError_t le = launch_kernel(indexer_tc_kernel<1, kMx, true>, dim3(seq.T * cl), dim3(TcWarps<1, kMx>::kThreads),
                                       smem, env.stream, true, cl, kmap, kmap2, qmap, p);
  if (le != cudaSuccess) return le;
  char buf[160];
  snprintf(buf, sizeof(buf), "indexer_topk_fused<%s>[cluster=%d,grid=%d]", kMx ? "mxfp8" : "e4m3", cl, seq.T * cl);
  *plan += buf;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_fused(const SeqArgs& seq, const IndexerArgs& a, int32_t K, int32_t* idx,
                                const LaunchEnv& env, std::string* plan, bool* unsupported, std::string* why) {
  *unsupported = true;
  if (seq.T == 0 || K < 1) return cudaSuccess;
  const bool tc_ok = a.e4m3 && a.H_I == kTcHeads && a.D_I == kTcDim && seq.page_size == kTcPage &&
                     (reinterpret_cast<uintptr_t>(a.k) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.q) % 16 == 0);
  // several queries of one sequence share their key reads in the chained plan
  if (!tc_ok || seq.q_per_seq > 1 || seq.T > env.num_sms) return cudaSuccess;
  const int cl = a.mx ? fused_cluster<true>(seq, env, kFusedMaxCluster) : fused_cluster<false>(seq, env, kFusedMaxCluster);
  // Measured on GB300: with one or two CTAs per query (a batch of >= num_sms / 4
  // queries) the fused kernel beats the chained indexer + Top-K (decode batch 64:
  // 81.0 vs 83.7 us a step); with more CTAs per query the selection's exchanges
  // between them cost more than the chained plan's score round trip (decode
  // batch 1: 25.9 vs 25.7 us; batch 4 at 131072 positions: 61.1 vs 55.8 us).
  if (cl < 1 || cl > kFusedMaxCluster) return cudaSuccess;
  *unsupported = false;
  return a.mx ? launch_fused<true>(seq, a, K, idx, cl, env, plan, why, unsupported)
              : launch_fused<false>(seq, a, K, idx, cl, env, plan, why, unsupported);
}

cudaError_t launch_indexer(const SeqArgs& seq, const IndexerArgs& a, const LaunchEnv& env,
                           std::string* plan, bool* unsupported, std::string* why) {
  *unsupported = false;
  if (seq.T == 0) {
    *plan += "indexer[empty]";
    return cudaSuccess;
  }
  const bool tc_ok = a.e4m3 && a.H_I == kTcHeads && a.D_I == kTcDim && seq.page_size == kTcPage &&
                     (reinterpret_cast<uintptr_t>(a.k) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.q) % 16 == 0);
  if (tc_ok) {
    if (a.mx) return launch_tc<1, true>(seq, a, env, plan, unsupported, why);
    const int qps = seq.q_per_seq;
    if (qps > 0 && qps % 4 == 0) return launch_tc<4>(seq, a, env, plan, unsupported, why);
    if (qps > 0 && qps % 2 == 0) return launch_tc<2>(seq, a, env, plan, unsupported, why);
    return launch_tc<1>(seq, a, env, plan, unsupported, why);
  }
  const size_t smem = (static_cast<size_t>(a.H_I) * a.D_I + a.H_I) * sizeof(float);
  if (smem > 200 * 1024) {
    *unsupported = true;
    *why = "indexer: H_I * D_I too large for the generic kernel";
    return cudaSuccess;
  }
  dim3 grid((seq.max_ctx + kGenThreads - 1) / kGenThreads, seq.T);
  const int fmt = a.mx ? 2 : (a.e4m3 ? 1 : 0);
  void (*kern)(SeqArgs, IndexerArgs) = fmt == 2 ? indexer_generic_kernel<2>
                                       : (fmt == 1 ? indexer_generic_kernel<1> : indexer_generic_kernel<0>);
  if (smem > 48 * 1024) {
    const cudaError_t ae = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (ae != cudaSuccess) return ae;
  }
  const cudaError_t le = launch_kernel(kern, grid, dim3(kGenThreads), smem, env.stream, true, 1, seq, a);
  if (le != cudaSuccess) return le;
  *plan += fmt == 2 ? "indexer_generic<mxfp8>" : (fmt == 1 ? "indexer_generic<e4m3>" : "indexer_generic<f32>");
  return cudaGetLastError();
}

}  // namespace dsa
