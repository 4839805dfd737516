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
//  * attn_tc48_kernel<kFp8> -- tensor-core path for H = 128, 512 + 64 dims, bf16
//    rows or 656-byte FP8 rows, 48-row tiles.  One CTA handles one query, one
//    half of the value dims (256 of 512) and one contiguous slice of the selected
//    rows; the CTA pair covering both value halves computes the same logits
//    (O[128 x 512] fp32 would fill all of TMEM, so each CTA keeps a [128 x 256]
//    accumulator).  FP8 codes are widened to bf16 exactly while gathering; the
//    per-row scale is applied to the latent part of the logit (latent and rope
//    logits accumulate in separate TMEM columns) and folded into P for P V, so
//    the FP8 path rounds nothing the bf16 path does not.  Layout and warp roles
//    are described above the kernel.
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
      // per-token scale at byte 512, or (per-128-tile rows) scale d / 128 at 512 + 4 (d / 128)
      const int si = kind == MlaKind::kFP8Tile ? d / 128 : 0;
      if (d < 512) return e4m3_to_float(row[d]) * reinterpret_cast<const float*>(row + 512)[si];
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
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescPV = make_idesc(kFmtBF16, kFmtBF16, false, true, kH, kDvHalf);
// Running max moved (and O rescaled) only when it grows by more than 2^64: P is
// bf16 and O, l fp32, whose ranges hold such factors with room to spare (P <=
// 2^64, O and l <= 2^64 x rows x max|row|), and a rescale stalls a softmax warp
// for ~2000 cycles, which a threshold of 2^8 met often in causal prefill.
constexpr float kRescaleThreshold = 64.0f;         // log2 units

struct TcAttnParams {
  SeqArgs seq;
  MlaArgs a;
  int32_t n_split;       // row slices per query
  int32_t rows_per_split;
  uint16_t* ws_o;        // [n_split, T, H, 512] bf16 partials (n_split > 1), each normalised by its own sum
  float* ws_lse;         // [n_split, T, H]
  uint64_t wait_limit_ns;   // bound of every pipeline wait
  uint32_t dbg_withhold;    // testing aid: producer warp 0 withholds its arrival on tile 0
};

// Byte offset of 16-byte chunk `ch` of tile row `r` in a 128B-swizzled K-major
// tile of `rows` rows: atom (64 values) major, then row, then swizzled chunk.
__device__ __forceinline__ uint32_t sw128_offset(int r, int ch, int rows) {
  return static_cast<uint32_t>((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}


// ---------------------------------------------------------------------------
// 48-row tiles: three stages for bf16 rows, two for FP8 rows.
//
// Producers (warps 0-11), bf16 rows: all twelve warps load every tile, four rows
// each (a warp issues cp.async copies at ~30 ns per instruction here, so the
// warps per tile set how fast it lands).  Lanes resolve the rows (index -> page
// -> cache row; the index is loaded one tile ahead) and, while the stage is
// still busy, ask L2 to fetch them; once it is free every lane copies its fixed
// 16-byte chunks of each row with cp.async into the 128B-swizzled K-major tile
// and moves on to the next tile without waiting: the copies arrive on the
// stage's barrier when they land (cp.async.mbarrier.arrive.noinc), so a warp
// keeps up to three tiles in flight.  Rows that select nothing are zeroed.  (On
// this GPU a tile::gather4 TMA producer reached ~12 GB/s per SM and cp.async
// gathers ~60 GB/s.)  FP8 rows with per-128 tile scales share this plan; their
// lanes load the codes into registers before the stage is free and widen them
// into the tile.  FP8 rows with one scale per row: two groups of six warps, 8
// rows per warp, each group owning one stage; a lane loads 16 codes of each of
// its warp's rows into registers before the stage is free, then widens them to
// bf16 into the tile; the rope goes by cp.async.
//
// MMA warps: warp 12 issues Q K^T_{j+1} (N = 48 rows) as soon as tile j+1 has
// landed and its logit buffer has been read, so it runs
// during the softmax of tile j; warp 13 issues P V_j (N = 256 value dims) as
// soon as P_j is written.  (One warp issuing both made a ready P V wait behind the issue
// of a Q K^T and vice versa: the issuing thread blocks until the tensor pipe
// has taken the instructions.)  An M=128
// K=16 step whose A operand (the query) sits in shared memory reads 6 KB of
// shared memory and takes ~53 clk, one with A in TMEM ~36 clk, so the first 320
// query dims live in TMEM.
//
// Softmax (warps 14-17): one thread per head (its TMEM lane), 48 logits a tile,
// running max moved (and O rescaled in TMEM) only when it grows by more than
// 2^64.
//
// bf16 rows -- TMEM: S double-buffered [0,48) and [48,96), Q [96,256), O
// [256,512); shared memory: query dims [320, 576) (64 KB) + three 54 KB tiles.
// Once Q K^T_j is complete, the 256 latent dims of tile j that this CTA's value
// half does not use are dead, and the softmax writes P_j there (128 x 48 bf16, 128B-swizzled K-major, the A operand of
// P V_j), so TMEM holds two logit buffers: Q K^T_{j+1} is issued as soon as
// tile j+1 lands, without waiting for the softmax to
// read S_j, and the tensor pipe does not idle across that hand-off (~700
// cycles a tile with one buffer).  The third stage hides the gather of a tile
// behind the work on the other two.  FP8 rows: see the T48 plan below.
constexpr int kBR48 = 48;
constexpr int kTile48Bytes = kBR48 * kDqk * 2;                 // 55296
constexpr int kT48Threads = 576;   // warps 0-11 producers, 12 Q K^T, 13 P V, 14-17 softmax
constexpr int kT48Mma = 12;        // Q K^T issuer; also allocates TMEM
constexpr int kT48Pv = 13;         // P V issuer
constexpr int kT48Soft = 14;       // first softmax warp
constexpr int kT48SmemBytes = 232448;
constexpr uint32_t kIdescS48 = make_idesc(kFmtBF16, kFmtBF16, false, false, kH, kBR48);

// Per row format.  bf16 rows: three stages; query dims [0, 320) in TMEM.
// FP8 rows: the latent codes are widened to bf16 exactly and the per-row scale
// is applied to the latent logits and folded into P, so the rope logits need
// their own 48 TMEM columns (Sr): the query keeps dims [0, 256) in TMEM and
// [256, 576) in shared memory (80 KB), which leaves room for two stages; the
// logits are single-buffered and P sits in TMEM.
//   bf16 TMEM: S0 [0,48), S1 [48,96), Q [96,256), O [256,512); P in the stage
//   FP8  TMEM: S [0,48), Sr [48,96), P [96,120), Q [128,256), O [256,512)
template <bool kFp8>
struct T48 {
  static constexpr int kStages = kFp8 ? 2 : 3;
  // bf16 rows: the twelve producer warps all load every tile (four rows each) and
  // run up to kStages tiles ahead, each lane's copies arriving on the stage's
  // barrier as they land; FP8 rows: one group of six warps per stage, each warp
  // converting its rows and waiting for its copies before it arrives
  static constexpr int kGroups = kFp8 ? kStages : 1;
  static constexpr bool kAsyncArrive = kGroups == 1;
  static constexpr int kProducers = 12 / kGroups;          // warps per tile
  static constexpr int kRows = kBR48 / kProducers;         // tile rows per producer warp
  // arrivals that complete a stage's barrier: one per warp (after its shared
  // stores), plus one per lane when its copies land (asynchronous arrival)
  static constexpr uint32_t kFullCount = kProducers * (kAsyncArrive ? 33 : 1);
  static constexpr int kQTmemDims = kFp8 ? 256 : 320;
  static constexpr int kQTmemSteps = kQTmemDims / 16;
  static constexpr int kQSmemAtoms = (kDqk - kQTmemDims) / 64;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQSmemAtoms * kH * 128;
  static constexpr int kOffMask = kOffKV + kStages * kTile48Bytes;     // uint16 [stages][producers]
  // FP8 rows: float [stages][48] row scales, then float [stages][48] their reciprocals
  static constexpr int kOffScale = kOffMask + 128;
  static constexpr int kOffBar = kOffScale + (kFp8 ? 2 * kStages * kBR48 * 4 : 0);
  // barriers: full[S], empty[S], sfull[2], sfree[2], pfull[S], ofull, drain
  static constexpr int kNumBars = 3 * kStages + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kUsed = kOffMisc + 16;                           // bytes used from the aligned base
  // the dynamic shared-memory base is re-aligned to 1024 B inside the kernel;
  // the rest of the allocation is slack for that (the kernel checks it sufficed)
  static constexpr int kSlack = kT48SmemBytes - kUsed;
  static constexpr uint32_t kColS = 0, kColSr = 48;
  static constexpr uint32_t kColP = 96, kColQ = kFp8 ? 128 : 96, kColO = 256;   // kColP: FP8 rows
  // bf16 rows: two logit buffers, P in the stage (the other value half's latent
  // dims, dead once Q K^T of the tile is complete) instead of TMEM
  static constexpr int kSBufs = kFp8 ? 1 : 2;
  static constexpr bool kPSmem = !kFp8;
  static_assert(kColQ + kQTmemDims / 2 <= kColO, "TMEM plan");
  static_assert(kFp8 ? (kColS + kBR48 <= kColSr && kColSr + kBR48 <= kColP && kColP + kBR48 / 2 <= kColQ)
                     : (kColS + kSBufs * kBR48 <= kColQ), "TMEM plan");
  static_assert(kStages * kProducers * 2 <= 128 && kSlack >= 128, "shared memory budget");
  static_assert(kGroups * kProducers == 12 && kProducers * kRows == kBR48, "producer warps");
};

// Q K^T of one 48-row tile (elected lane of the MMA warp).  FP8 rows: the 32
// latent steps accumulate into S, the 4 rope steps into Sr.
template <bool kFp8>
__device__ __forceinline__ void t48_issue_s(uint32_t tmem, uint32_t scol, uint64_t dq0, uint64_t dk) {
  using C = T48<kFp8>;
#pragma unroll
  for (int kk = 0; kk < kDqk / 16; ++kk) {
    const uint64_t db = dk + static_cast<uint64_t>(((kk >> 2) * kBR48 * 128 + (kk & 3) * 32) >> 4);
    const bool rope = kFp8 && kk >= kDv / 16;
    const uint32_t acc = (kk == 0 || (kFp8 && kk == kDv / 16)) ? 0u : 1u;
    const uint32_t d = tmem + (rope ? C::kColSr : scol);
    if (kk < C::kQTmemSteps) {
      umma_f16_tmem_a(d, tmem + C::kColQ + kk * 8, db, kIdescS48, acc);
    } else {
      const int qk = kk - C::kQTmemSteps;
      const uint64_t da = dq0 + static_cast<uint64_t>(((qk >> 2) * kH * 128 + (qk & 3) * 32) >> 4);
      umma_f16(d, da, db, kIdescS48, acc);
    }
  }
}

// kTile: FP8 rows with one power-of-two scale per 128 latent dims, widened to
// bf16 as code * scale by the producers (exact); the rest runs the bf16 plan.
template <bool kFp8, bool kTile = false>
__global__ void __launch_bounds__(kT48Threads, 1) attn_tc48_kernel(TcAttnParams p) {
  using C = T48<kFp8>;
  constexpr int S = C::kStages;
  // No grid_dep_wait() here: setup and the query staging overlap the kernel
  // before (Top-K), which lets this grid launch early; the producers wait for
  // it before they read the selected indices.  The kernel after (the combine,
  // or the next step's indexer) may launch at once too: each waits for this
  // grid before it reads anything this grid writes.
  grid_dep_launch();
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // re-aligned by pointer arithmetic on the shared array, so that the compiler
  // keeps every access through `sm` in the shared window
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  if (sm - sm_raw > C::kSlack) {   // block-uniform: the re-aligned layout would not fit
    if (threadIdx.x == 0) atomicOr(&g_status_attn, kDevConfig);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* full = bars;            // [S] tile landed (one arrival per warp of the stage's group)
  uint64_t* empty = bars + S;       // [S] tile consumed by P V
  uint64_t* sfull = bars + 2 * S;   // [2] logits ready (per logit buffer)
  uint64_t* sfree = sfull + 2;      // [2] logits read by the softmax (buffer reusable)
  uint64_t* pfull = sfull + 4;      // [S] P of the stage's tile written
  uint64_t* ofull = pfull + S;      // every MMA done
  uint64_t* drain = ofull + 1;      // both issuing warps' MMAs complete (teardown)
  const uint64_t wlim = p.wait_limit_ns;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile uint16_t* mask16 = reinterpret_cast<volatile uint16_t*>(sm + C::kOffMask);   // [stage][warp]
  volatile float* row_scale = reinterpret_cast<volatile float*>(sm + C::kOffScale);    // [stage][48], FP8 rows
  volatile float* row_rcp = row_scale + S * kBR48;                                     // 1 / scale (0 for none)

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
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], C::kFullCount);
      mbar_init(&empty[i], 1);
      mbar_init(&pfull[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], 128);
    }
    mbar_init(ofull, 1);
    mbar_init(drain, 2);
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
    const uint32_t qbase = smem_u32(sm + C::kOffQ);
    constexpr int kChunks = (kDqk - C::kQTmemDims) / 8;
    for (int i = threadIdx.x - kT48Mma * 32; i < kH * kChunks; i += kQBarThreads) {
      const int h = i / kChunks, ch = i % kChunks;
      cp_async16(qbase + sw128_offset(h, ch, kH), qg + h * kDqk + C::kQTmemDims + ch * 8);
    }
    cp_async_commit();
  }
  if (warp >= kT48Soft) {
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint4* qrow = reinterpret_cast<const uint4*>(qg + h * kDqk);
    // every 128-byte line of this head's TMEM part requested from L2 at once: the
    // blocks below then wait one L2 round trip each instead of one HBM round trip
#pragma unroll
    for (int blk = 0; blk < C::kQTmemDims / 64; ++blk) prefetch_l2(qrow + blk * 8);
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
  if (warp >= kT48Mma) {
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    named_bar_sync(kQBar, kQBarThreads);
    tc_fence_after();
  }

  if (warp < C::kProducers * C::kGroups) {
    // ------------------------------------------------ producers: group g loads tiles j = g mod
    // kGroups into stage j mod S; warp w of the group copies tile rows [w*kRows, (w+1)*kRows)
    grid_dep_wait();   // the selected indices come from the kernel before
    constexpr int kRows = C::kRows;
    const int grp = warp / C::kProducers, pw = warp % C::kProducers;
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
    // the selected position of this lane's row of tile j (lanes < kRows), or -1;
    // loaded one tile ahead of its use
    auto load_pos = [&](int j) -> int {
      const int gi = r0 + j * kBR48 + pw * kRows + lane;
      return (lane < kRows && gi < r1) ? __ldg(idx + gi) : -1;
    };
    int pos_next = load_pos(grp);
    for (int j = grp; j < ntiles; j += C::kGroups) {
      const int st = j % S;
      const uint32_t stage = smem_u32(sm + C::kOffKV + st * kTile48Bytes);
      const int pos = pos_next;
      pos_next = load_pos(j + C::kGroups);
      int64_t my_row = -1;
      if (pos >= 0) {
        if (pos > qp)
          atomicOr(&g_status_attn, kDevBadIndex);
        else
          my_row = phys_row(bt, pos, p.seq.page_size, p.seq.n_pages, &g_status_attn);
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, my_row >= 0) & ((1u << kRows) - 1u);
      // every row number first: a shuffle queues behind earlier cp.async copies
      int32_t rows[kRows];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) rows[rr] = __shfl_sync(0xffffffffu, static_cast<int32_t>(my_row), rr);
      // FP8 rows: the codes (16 per lane and row) and the row scales are loaded
      // into registers while the stage may still be busy
      uint4 raw[(kFp8 || kTile) ? kRows : 1];
      float tsc[kTile ? kRows : 1];   // per-128-tile rows: the scale of this lane's tile (lane / 8)
      float my_scale = 0.f;
      if constexpr (kFp8 || kTile) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr)
          raw[rr] = rows[rr] >= 0 ? ld_global_nc_v4(kv + static_cast<int64_t>(rows[rr]) * p.a.row_bytes + lane * 16)
                                  : make_uint4(0u, 0u, 0u, 0u);
      }
      if constexpr (kFp8) {
        if (my_row >= 0) my_scale = __ldg(reinterpret_cast<const float*>(kv + my_row * p.a.row_bytes + kDv));
      }
      if constexpr (kTile) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr)
          tsc[rr] = rows[rr] >= 0 ? __ldg(reinterpret_cast<const float*>(kv + static_cast<int64_t>(rows[rr]) *
                                                                                   p.a.row_bytes + kDv) + (lane >> 3))
                                  : 0.f;
      }
      if (j >= S) {
        if constexpr (!kFp8 && !kTile) {
          // the stage is still busy: have L2 fetch this warp's rows (9 lines of 128 B each) meanwhile
#pragma unroll
          for (int k = 0; k < (kRows * 9 + 31) / 32; ++k) {
            const int i = lane + 32 * k;
            const int64_t prow = __shfl_sync(0xffffffffu, my_row, min(i / 9, kRows - 1));
            if (i < kRows * 9 && prow >= 0) prefetch_l2(kv + prow * p.a.row_bytes + (i % 9) * 128);
          }
        }
        const bool ok = mbar_wait(&empty[st], ((j / S) - 1) & 1, &g_status_attn, abort_flag, wlim);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) mask16[st * C::kProducers + pw] = static_cast<uint16_t>(bits);
      if (kFp8 && lane < kRows) {
        row_scale[st * kBR48 + pw * kRows + lane] = my_scale;
        row_rcp[st * kBR48 + pw * kRows + lane] = my_scale > 0.f ? 1.f / my_scale : 0.f;
      }
      if constexpr (!kFp8 && !kTile) {
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
      } else {
        // FP8 rows (656 B: 512 e4m3 codes, fp32 scale, 12 reserved, 64 bf16 rope):
        // the rope is copied as it is (chunks 64-71, lanes 0-7); the latent codes
        // are widened to bf16 exactly into chunks 2*lane, 2*lane+1 (the row scale
        // is applied to the logits and to P by the softmax)
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const int r = pw * kRows + rr;
          const int64_t prow = rows[rr];
          const uint32_t drow = stage + static_cast<uint32_t>(r * 128);
          if (lane < 8) {
            const uint32_t dst = drow + 8 * kBR48 * 128 + static_cast<uint32_t>(((lane & 7) ^ (r & 7)) << 4);
            if (prow >= 0)
              cp_async16(dst, kv + prow * p.a.row_bytes + 528 + lane * 16);
            else
              st_shared_v4(dst, 0u, 0u, 0u, 0u);
          }
          const uint32_t w[4] = {raw[rr].x, raw[rr].y, raw[rr].z, raw[rr].w};
          const float sc = kTile ? tsc[rr] : 1.f;   // per-token rows: the scale goes to the logits and P
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w[k] & 0xFFFFu));
            const float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w[k] >> 16));
            o[2 * k] = pack_bf16x2(lo.x * sc, lo.y * sc);
            o[2 * k + 1] = pack_bf16x2(hi.x * sc, hi.y * sc);
          }
          // chunk ch = 2*lane + e of row r: atom ch >> 3, swizzled position (ch & 7) ^ (r & 7)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ch = 2 * lane + e;
            const uint32_t dst = drow + static_cast<uint32_t>((ch >> 3) * kBR48 * 128) +
                                 static_cast<uint32_t>(((ch & 7) ^ (r & 7)) << 4);
            st_shared_v4(dst, o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
          }
        }
      }
      if (p.dbg_withhold && warp == 0 && j == 0) continue;   // testing aid: this stage never completes
      if constexpr (C::kAsyncArrive) {
        // each lane's copies arrive when they land; lane 0 arrives for the warp's
        // shared stores (row mask, zeroed rows).  The MMA warps fence the async
        // proxy after their waits.
        cp_async_mbar_arrive(&full[st]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      } else {
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[st]);
      }
    }
    // nothing of this warp in flight when the CTA tears down
    cp_async_commit();
    cp_async_wait<0>();
  } else if (warp == kT48Mma || warp == kT48Pv) {
    // ------------------------------------------------ MMA issuers (whole warp, elected lane issues)
    // Bounded waits on the suspending try_wait: the issuing warps share their
    // sub-partitions with softmax warps, whose issue slots a spinning poll took
    // (prefill attention 2 % slower with test_wait spins).
    auto poll = [&](uint64_t* bar, uint32_t parity) -> bool {
      const uint32_t addr = smem_u32(bar);
      uint64_t t0 = 0;
      for (uint32_t it = 0;; ++it) {
        if (__shfl_sync(0xffffffffu, mbar_try_wait(addr, parity) ? 1 : 0, 0)) return true;
        if ((it & 255u) == 255u) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) return false;
          const uint64_t now = __shfl_sync(0xffffffffu, globaltimer_ns(), 0);
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > wlim) {
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
      const uint64_t dq0 = make_sdesc(smem_u32(sm + C::kOffQ), 16, 1024, kLayoutSw128);
      const uint64_t dk0 = make_sdesc(smem_u32(sm + C::kOffKV), 16, 1024, kLayoutSw128);
      for (int j = 0; j < ntiles; ++j) {
        // Q K^T_j: tile j has landed and the softmax has read the logits last
        // held by this buffer (S_{j - kSBufs})
        const int sb = j % C::kSBufs;
        if (j >= C::kSBufs && !poll(&sfree[sb], ((j / C::kSBufs) - 1) & 1)) break;
        // (Q K^T_j used to wait for P V_{j-2} to be queued as well; with the
        // softmax as short as it is now, letting it go as soon as its buffer and
        // tile are ready measured 0.7 % faster at decode batch 64.)
        if (!poll(&full[j % S], (j / S) & 1)) break;
        tc_fence_after();
        fence_proxy_async_smem();   // the copies that landed are visible to the tensor core
        if (elect_one()) {
          t48_issue_s<kFp8>(tmem, C::kColS + sb * kBR48, dq0,
                            dk0 + static_cast<uint64_t>(((j % S) * kTile48Bytes) >> 4));
          umma_commit(&sfull[sb]);
        }
        __syncwarp();
      }
    } else {
      const uint64_t dv0 = make_sdesc(smem_u32(sm + C::kOffKV) + c * 4 * kBR48 * 128, kBR48 * 128, 1024, kLayoutSw128);
      // bf16 rows: P_j in stage j mod S, where the other value half's latent dims were
      const uint64_t dp0 = make_sdesc(smem_u32(sm + C::kOffKV) + (1 - c) * 4 * kBR48 * 128, 16, 1024, kLayoutSw128);
      for (int j = 0; j < ntiles; ++j) {
        // P V_j as soon as P_j is written.  Its commit also covers Q K^T_j (complete
        // before the softmax wrote P_j), so empty[st] frees the whole stage and
        // tells the softmax that O holds P V_j; ofull marks every MMA of the CTA done.
        const int st = j % S;
        if (!poll(&pfull[st], (j / S) & 1)) break;
        tc_fence_after();
        fence_proxy_async_smem();
        const uint64_t dv = dv0 + static_cast<uint64_t>((st * kTile48Bytes) >> 4);
        const uint64_t dp = dp0 + static_cast<uint64_t>((st * kTile48Bytes) >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBR48 / 16; ++kk) {
            const uint64_t db = dv + static_cast<uint64_t>((kk * 16 * 128) >> 4);
            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
            if constexpr (C::kPSmem)
              umma_f16(tmem + C::kColO, dp + static_cast<uint64_t>((kk * 32) >> 4), db, kIdescPV, acc);
            else
              umma_f16_tmem_a(tmem + C::kColO, tmem + C::kColP + kk * 8, db, kIdescPV, acc);
          }
          umma_commit(&empty[st]);
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
    // FP8 rows: the stage's row scales and their reciprocals (shared addresses)
    const uint32_t scale_addr = smem_u32(sm + C::kOffScale);
    const uint32_t rcp_addr = scale_addr + S * kBR48 * 4;
    float m = -INFINITY, l = 0.f, l32 = 0.f;
    bool ok = true;
    // P_j goes to stage j mod S, where the latent dims of the other value half were
    const uint32_t p_row = smem_u32(sm + C::kOffKV) + static_cast<uint32_t>((1 - c) * 4 * kBR48 * 128 + h * 128);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % S;
      const int sb = j % C::kSBufs;
      const uint32_t scol = C::kColS + sb * kBR48;
      ok = mbar_wait(&sfull[sb], (j / C::kSBufs) & 1, &g_status_attn, abort_flag, wlim);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // the producers' row mask is ordered by their release on full[st] (still the
      // current phase: the stage is refilled only after this tile's P V)
      ok = mbar_wait(&full[st], (j / S) & 1, &g_status_attn, abort_flag, wlim);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float x[kBR48];
      {
        uint32_t s0[32], s1[16];
        tmem_ld32(tmem + lane_off + scol, s0);
        tmem_ld16(tmem + lane_off + scol + 32, s1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kBR48; ++i) x[i] = __uint_as_float(i < 32 ? s0[i & 31] : s1[(i - 32) & 15]);
      }
      if constexpr (kFp8) {
        // logit = row scale * latent part + rope part (packed fmas; the row scales
        // as 16-byte shared loads)
#pragma unroll
        for (int c16 = 0; c16 < kBR48 / 16; ++c16) {
          uint32_t r16[16];
          tmem_ld16(tmem + lane_off + C::kColSr + c16 * 16, r16);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 sc = ld_shared_v4(scale_addr + static_cast<uint32_t>((st * kBR48 + c16 * 16 + 4 * q) * 4));
            const int i = c16 * 16 + 4 * q;
            float y0 = __uint_as_float(r16[4 * q]), y1 = __uint_as_float(r16[4 * q + 1]);
            float y2 = __uint_as_float(r16[4 * q + 2]), y3 = __uint_as_float(r16[4 * q + 3]);
            fma2(y0, y1, __uint_as_float(sc.x), __uint_as_float(sc.y), x[i], x[i + 1]);
            fma2(y2, y3, __uint_as_float(sc.z), __uint_as_float(sc.w), x[i + 2], x[i + 3]);
            x[i] = y0;
            x[i + 1] = y1;
            x[i + 2] = y2;
            x[i + 3] = y3;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sfree[sb]);
      uint64_t vmask = 0;
      if constexpr (C::kProducers == 12 && C::kRows == 4) {
        // bf16 rows: the twelve 4-bit masks as three 8-byte loads (each u16 holds
        // its warp's bits in its low nibble); a full tile needs no compaction
        const volatile uint64_t* m64 = reinterpret_cast<const volatile uint64_t*>(mask16 + st * C::kProducers);
        const uint64_t w0 = m64[0], w1 = m64[1], w2 = m64[2];
        constexpr uint64_t kAll = 0x000F000F000F000Full;
        if (((w0 ^ kAll) | (w1 ^ kAll) | (w2 ^ kAll)) == 0) {
          vmask = (1ull << kBR48) - 1u;
        } else {
          auto nib = [](uint64_t w) -> uint64_t {
            w &= kAll;
            w = (w | (w >> 12)) & 0x000000FF000000FFull;
            return (w | (w >> 24)) & 0xFFFFull;
          };
          vmask = nib(w0) | (nib(w1) << 16) | (nib(w2) << 32);
        }
      } else {
#pragma unroll
        for (int w = 0; w < C::kProducers; ++w)
          vmask |= static_cast<uint64_t>(mask16[st * C::kProducers + w]) << (w * C::kRows);
      }
      // Rows that select nothing are set to -inf (the selects skipped when every
      // row of the tile is valid: CTA-uniform); the row maximum is taken over four
      // independent partial maxima of three-input maxes.  The logits stay unscaled
      // here: fl(x * s) is monotone in x, so the maximum of the scaled logits is
      // the scaled maximum, and the exponent below is one packed fma x * s - m.
      if (vmask != (1ull << kBR48) - 1u) {
#pragma unroll
        for (int i = 0; i < kBR48; ++i) x[i] = ((vmask >> i) & 1u) ? x[i] : -INFINITY;
      }
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < kBR48; i += 2) mq[(i >> 1) & 3] = fmax3(mq[(i >> 1) & 3], x[i], x[i + 1]);
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      const float mloc = mx * sl2;
      // P V_{j-1} is done once it has freed its stage: empty[(j-1) mod S] in the
      // phase of tile j-1 (the phase before it completed when tile j-1 was
      // loaded, the one after needs P_{j-1+S}, so a parity wait cannot alias)
      const int stp = (j + S - 1) % S;
      const uint32_t par_prev = ((j - 1) / S) & 1;
      const float m_new = fmaxf(m, mloc);
      const bool need = m_new > m + kRescaleThreshold;
      if (j >= 1 && __any_sync(0xffffffffu, need)) {
        // O is rescaled: P V_{j-1} must have written it
        ok = mbar_wait(&empty[stp], par_prev, &g_status_attn, abort_flag, wlim);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
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
        tmem_st_wait();   // O rescaled before P V_j may accumulate into it
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
      if constexpr (!kFp8) {
        // bf16 rows: exponents x * s - m as packed fmas, sums over pairs, two pairs
        // of running sums each of the rounded weights (what P V multiplies) and of
        // the exact ones
        float sr[4] = {0.f, 0.f, 0.f, 0.f}, se[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBR48 / 2; ++i) {
          float d0 = -msub, d1 = -msub;
          fma2(d0, d1, x[2 * i], x[2 * i + 1], sl2, sl2);
          const float p0 = fast_exp2(d0), p1 = fast_exp2(d1);
          const int a = 2 * (i & 1);
          add2(se[a], se[a + 1], se[a], se[a + 1], p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
          add2(sr[a], sr[a + 1], sr[a], sr[a + 1], __uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xFFFF0000u));
        }
        psum = (sr[0] + sr[1]) + (sr[2] + sr[3]);
        psum32 = (se[0] + se[1]) + (se[2] + se[3]);
      } else {
        // FP8 rows: P V runs on the unscaled codes, so the row scale is folded into
        // P, and the denominator takes the rounded weights times the reciprocal
        // scale (the producers' 1 / scale, 0 for a row without one); packed ops,
        // scales and reciprocals as 16-byte shared loads, four logits at a time
        float sr[2] = {0.f, 0.f}, se[2] = {0.f, 0.f};
#pragma unroll
        for (int c4 = 0; c4 < kBR48 / 4; ++c4) {
          const uint32_t off = static_cast<uint32_t>((st * kBR48 + 4 * c4) * 4);
          const uint4 sc = ld_shared_v4(scale_addr + off), rc = ld_shared_v4(rcp_addr + off);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int i = 2 * c4 + q;   // logit pair
            float d0 = -msub, d1 = -msub;
            fma2(d0, d1, x[2 * i], x[2 * i + 1], sl2, sl2);
            const float p0 = fast_exp2(d0), p1 = fast_exp2(d1);
            add2(se[0], se[1], se[0], se[1], p0, p1);
            float w0, w1;
            mul2(w0, w1, p0, p1, __uint_as_float(q ? sc.z : sc.x), __uint_as_float(q ? sc.w : sc.y));
            pk[i] = pack_bf16x2(w0, w1);
            fma2(sr[0], sr[1], __uint_as_float(pk[i] << 16), __uint_as_float(pk[i] & 0xFFFF0000u),
                 __uint_as_float(q ? rc.z : rc.x), __uint_as_float(q ? rc.w : rc.y));
          }
        }
        psum = sr[0] + sr[1];
        psum32 = se[0] + se[1];
      }
      l += psum;
      l32 += psum32;
      if constexpr (C::kPSmem) {
        // row h of the 128B-swizzled K-major P tile: 16-byte chunk q at q ^ (h & 7)
        const uint32_t prow = p_row + static_cast<uint32_t>(st * kTile48Bytes);
#pragma unroll
        for (int q = 0; q < kBR48 / 8; ++q)
          st_shared_v4(prow + static_cast<uint32_t>((q ^ (h & 7)) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                       pk[4 * q + 3]);
        fence_proxy_async_smem();   // visible to the tensor core's P V_j
      } else {
        if (j >= 1) {
          // P (one TMEM buffer) was read by P V_{j-1}
          ok = mbar_wait(&empty[stp], par_prev, &g_status_attn, abort_flag, wlim);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        uint32_t pa[16], pb[8];
#pragma unroll
        for (int i = 0; i < 16; ++i) pa[i] = pk[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) pb[i] = pk[16 + i];
        tmem_st16(tmem + lane_off + C::kColP, pa);
        tmem_st8(tmem + lane_off + C::kColP + 16, pb);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&pfull[st]);
    }
    if (ok) {
      ok = mbar_wait(ofull, 0, &g_status_attn, abort_flag, wlim);
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

  if (warp == kT48Mma || warp == kT48Pv) {
    // every MMA either issuing warp started has finished before TMEM is released
    // (after an abort, some may still be running)
    if (elect_one()) umma_commit(drain);
    __syncwarp();
    mbar_drain(drain, 0, &g_status_attn, wlim);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kT48Mma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merges row slices: out[t,h,:] = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max_s lse_s);
// lse = max + log sum_s w_s.  The partials O_s are bf16 rows, each normalised by
// its own slice's sum.  A CTA takes HPC heads of one query with SW warps per head:
// warp w of a head takes the slices w, w + SW, w + 2 SW, ..., eight at a time with
// all of their row and LSE loads in flight together; lane l owns the value dims
// [8l, 8l + 8) and [256 + 8l, 256 + 8l + 8), so each load instruction reads 512
// contiguous bytes.  A head's warps meet in shared memory with their running
// (max, sum, weighted row), and its threads write the output four dims at a time.
constexpr int kCombineBatch = 8;   // slices per warp per round trip
template <int SW, int HPC>
__global__ void __launch_bounds__(32 * SW * HPC)
    attn_combine_kernel(const uint16_t* ws_o, const float* ws_lse, int n_split, int T,
                        __nv_bfloat16* out, float* lse_out) {
  grid_dep_launch();   // the next kernel waits for this grid before it uses out
  grid_dep_wait();
  constexpr int H = kH;
  __shared__ float s_acc[SW * HPC][16][32];   // [warp][value slot][lane]
  __shared__ float s_m[SW * HPC], s_l[SW * HPC];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = warp / SW, sv = warp % SW;   // head within the CTA, slice phase
  const int h = blockIdx.y * HPC + hl;
  const int64_t th = static_cast<int64_t>(t) * H + h;
  const int64_t slice_stride = static_cast<int64_t>(T) * H * (kDv / 8);   // in 16-byte vectors
  const uint4* src = reinterpret_cast<const uint4*>(ws_o) + th * (kDv / 8) + lane;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int s0 = sv; s0 < n_split; s0 += SW * kCombineBatch) {
    const int nb = min(kCombineBatch, (n_split - s0 + SW - 1) / SW);   // slices s0 + u*SW, u < nb
    uint4 v[kCombineBatch][2];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (u < nb) {
        v[u][0] = __ldcs(src + (s0 + u * SW) * slice_stride);
        v[u][1] = __ldcs(src + (s0 + u * SW) * slice_stride + kDv / 16);
      }
    }
    const float ls =
        lane < nb ? ws_lse[(static_cast<int64_t>(s0 + lane * SW) * T + t) * H + h] : -INFINITY;
    float mb = ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float m_new = fmaxf(m, mb);
    // earlier batches rescaled to the new maximum (all zero while m is -inf)
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
#pragma unroll
  for (int k = 0; k < 16; ++k) s_acc[warp][k][lane] = acc[k];
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  __syncthreads();
  const int w0 = hl * SW;   // the head's first warp
  float mm = s_m[w0];
#pragma unroll
  for (int w = 1; w < SW; ++w) mm = fmaxf(mm, s_m[w0 + w]);
  float fw[SW], ll = 0.f;
#pragma unroll
  for (int w = 0; w < SW; ++w) {
    fw[w] = (s_m[w0 + w] == -INFINITY) ? 0.f : __expf(s_m[w0 + w] - mm);
    ll = fmaf(fw[w], s_l[w0 + w], ll);
  }
  const int i0 = threadIdx.x - w0 * 32;   // thread within the head's warps
  if (i0 == 0 && lse_out) lse_out[th] = ll > 0.f ? mm + logf(ll) : -INFINITY;
  const float inv = ll > 0.f ? 1.f / ll : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(out + th * kDv);
  // quad q holds dims [4q, 4q + 4): lane (q mod 64) / 2 of the warps, slots
  // 8 * (q / 64) + 4 * (q mod 2) .. + 3
#pragma unroll
  for (int q = i0; q < kDv / 4; q += 32 * SW) {
    const int src_lane = (q & 63) >> 1, k0 = 8 * (q >> 6) + 4 * (q & 1);
    float r[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < SW; ++w) x = fmaf(fw[w], s_acc[w0 + w][k0 + c][src_lane], x);
      r[c] = x * inv;
    }
    dst[q] = make_uint2(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]));
  }
}

// Launches the slice merge for T queries.  While the (query, head) pairs are no
// more than the SMs, four warps per head and one head per CTA, so that the loads
// spread over as many SMs as there are pairs; otherwise two heads per CTA with
// enough warps per head (1, 2 or 4) that each takes one batch of kCombineBatch
// slices.
cudaError_t launch_combine(const uint16_t* ws_o, const float* ws_lse, int n_split, int T,
                           __nv_bfloat16* out, float* lse_out, const LaunchEnv& env) {
  const int64_t pairs = static_cast<int64_t>(T) * kH;
  const int need = (n_split + kCombineBatch - 1) / kCombineBatch;
#define DSA_COMBINE(SW_, HPC_)                                                                           \
  launch_kernel(attn_combine_kernel<SW_, HPC_>, dim3(T, kH / (HPC_)), dim3(32 * (SW_) * (HPC_)), 0,      \
                env.stream, true, 1, ws_o, ws_lse, n_split, T, out, lse_out)
  if (pairs <= env.num_sms) return DSA_COMBINE(4, 1);
  if (need > 2) return DSA_COMBINE(4, 2);
  if (need > 1) return DSA_COMBINE(2, 2);
  return DSA_COMBINE(1, 2);
#undef DSA_COMBINE
}

bool tc_supported(const SeqArgs& seq, const MlaArgs& a) {
  if (a.H != kH || a.d_latent != kDv || a.d_rope != kDqk - kDv) return false;
  if (a.kind == MlaKind::kF32) return false;
  if (a.kind == MlaKind::kBF16 && a.row_bytes % 16 != 0) return false;
  if ((a.kind == MlaKind::kFP8Row || a.kind == MlaKind::kFP8Tile) && a.row_bytes % 16 != 0) return false;
  if (reinterpret_cast<uintptr_t>(a.kv) % 16 || reinterpret_cast<uintptr_t>(a.q) % 16 ||
      reinterpret_cast<uintptr_t>(a.out) % 16)
    return false;
  (void)seq;
  return true;
}

// Row slices per query: fill the GPU with (query, half, slice) CTAs, at least
// 4 tiles (128 rows) per slice, at most 64 slices.
int choose_split(const SeqArgs& seq, const MlaArgs& a, int num_sms) {
  // at least two 48-row tiles per slice: every slice stages the whole query, so
  // thinner slices lose
  const int min_rows = 2 * kBR48;
  const int max_split = std::min(64, std::max(1, (a.K + min_rows - 1) / min_rows));
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
    const bool tile = a.kind == MlaKind::kFP8Tile;
    const int tile_rows = kBR48;
    int split = choose_split(seq, a, env.num_sms);
    if (split > 1 && (workspace == nullptr || ws_bytes < attn_workspace_bytes(seq, a, env.num_sms)))
      split = 1;  // no room for partials: one slice per query
    const int rps = ((a.K + split - 1) / split + tile_rows - 1) / tile_rows * tile_rows;
    split = (a.K + rps - 1) / rps;  // every slice non-empty
    TcAttnParams p{seq, a, split, rps, nullptr, nullptr, kWaitLimitNs, 0u};
    debug_wait_state(&p.wait_limit_ns, &p.dbg_withhold);
    if (split > 1) {
      const size_t o = static_cast<size_t>(split) * seq.T * kH * kDv * sizeof(uint16_t);
      p.ws_o = static_cast<uint16_t*>(workspace);
      p.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o + 255) / 256) * 256);
    }
    void (*kern)(TcAttnParams) = fp8 ? attn_tc48_kernel<true> : (tile ? attn_tc48_kernel<false, true>
                                                                          : attn_tc48_kernel<false>);
    const cudaError_t attr_err = ensure_smem_limit(reinterpret_cast<const void*>(kern), kT48SmemBytes, env.device);
    if (attr_err != cudaSuccess) return attr_err;
    const int grid = seq.T * split * 2;
    const cudaError_t le = launch_kernel(kern, dim3(grid), dim3(kT48Threads), kT48SmemBytes, env.stream, true, 1, p);
    if (le != cudaSuccess) return le;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    char buf[128];
    snprintf(buf, sizeof(buf), "attn_tc<%s>[split=%d,grid=%d]", fp8 ? "fp8x48" : (tile ? "fp8t128x48" : "bf16x48"),
             split, grid);
    *plan += buf;
    if (split > 1) {
      e = launch_combine(static_cast<const uint16_t*>(p.ws_o), static_cast<const float*>(p.ws_lse), split, seq.T,
                         static_cast<__nv_bfloat16*>(a.out), a.lse, env);
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
  if (smem > 48 * 1024) {
    const cudaError_t ae = cudaFuncSetAttribute(attn_generic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(smem));
    if (ae != cudaSuccess) return ae;
  }
  dim3 grid(a.H, seq.T);
  const cudaError_t le = launch_kernel(attn_generic_kernel, grid, dim3(kGenThreads), smem, env.stream, true, 1, seq, a);
  if (le != cudaSuccess) return le;
  *plan += "attn_generic";
  return cudaGetLastError();
}

}  // namespace dsa
