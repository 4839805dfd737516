// Per-query Top-K over the causal history (step 2 of the DSA path).
//
// "Large Language Model Inference Acceleration in Practice", section 1.2: the
// lightning indexer selects the Top-K most relevant historical positions for the
// current query.  For query t with history n = q_pos[t] + 1 the kernel returns
// the min(K, n) positions with the largest fp32 scores, ties to the lower
// position, as an ascending list followed by -1 padding.
//
// Exact radix select:
//  * a query's history is split into contiguous slices over the CTAs of a
//    thread-block cluster (1 to 8 CTAs of 512 threads), each slice's scores
//    turned into order-preserving uint32 keys (-0.0 folded onto +0.0) and cached
//    in that CTA's shared memory;
//  * up to four 8-bit digit passes narrow the K-th largest key: every CTA builds
//    the histogram of its slice (one private histogram per warp over the warp's
//    contiguous range, four keys per thread per step, then summed), and after
//    one cluster barrier every CTA reads the cluster's histograms through
//    distributed shared memory and picks the same digit by itself (histograms
//    alternate between two buffers, so a pass needs no second barrier before the
//    next one overwrites them); a pass stops early when the bucket holding the
//    K-th key is taken whole;
//  * an ordered compaction keeps every key above the threshold and, in position
//    order, the first `remaining` keys equal to it.  Each warp's own histograms
//    give its counts above and on the threshold, and the other slices'
//    histograms (read in every pass anyway) give the counts of the slices before
//    this one, so no further exchange is needed: a scan over warps gives each
//    warp its offsets, and within a warp ballots over 32 consecutive keys give
//    each lane its slot, so the output comes out in ascending order.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

DSA_DEFINE_STATUS_WORD(topk)

namespace dsa {
namespace {

namespace cg = cooperative_groups;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMinSliceKeys = 1024;     // smallest history slice worth a CTA
constexpr int kCacheKeys = 48 * 1024;   // shared-memory key cache per CTA (192 KB)

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;  // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkArgs {
  const float* scores;
  int64_t ld;
  const int32_t* q_pos;
  int32_t max_ctx;
  int32_t K;
  int32_t* idx;
  int32_t cache_keys;  // keys cached per CTA in dynamic smem (0 = none)
  int32_t T;
};

// Exclusive scans over the warps of two per-warp values at once: every thread
// gets its warp's two offsets.  Uses `buf` [2][kWarps + 1] and two __syncthreads.
__device__ __forceinline__ void warp_offsets2(uint32_t c0, uint32_t c1, uint32_t (*buf)[kWarps + 1],
                                              uint32_t* excl0, uint32_t* excl1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    buf[0][warp] = c0;
    buf[1][warp] = c1;
  }
  __syncthreads();
  if (warp < 2) {
    const uint32_t v = lane < kWarps ? buf[warp][lane] : 0u;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane < kWarps) buf[warp][lane] = inc - v;
  }
  __syncthreads();
  *excl0 = buf[0][warp];
  *excl1 = buf[1][warp];
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
  grid_dep_wait();
  // The attention kernel that follows may start now: it stages its query and
  // waits for this grid before it reads the indices.
  grid_dep_launch();
  extern __shared__ uint32_t keys_s[];
  __shared__ uint32_t hist2[2][256];    // this CTA's slice (pass parity)
  __shared__ uint32_t whist[kWarps][256];   // per-warp partial histograms
  __shared__ uint32_t ghist[256];       // the cluster's sum
  __shared__ uint32_t scan_buf[2][kWarps + 1];
  __shared__ uint32_t s_digit, s_rem, s_bucket;
  // keys of the slices before this one (lower cluster ranks): above the
  // threshold, and equal to it -- read off their histograms, pass by pass
  __shared__ uint32_t s_gt_before, s_eq_before;

  cg::cluster_group cluster = cg::this_cluster();
  const int CL = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  // clusters take queries last-first: with causal histories (prefill) the longest
  // histories start first and the short ones fill the tail of the launch
  const int t = a.T - 1 - static_cast<int>(blockIdx.x) / CL;
  const int tid = threadIdx.x, lane = tid & 31;
  int qp = __ldg(a.q_pos + t);
  if (qp < 0 || qp >= a.max_ctx) {
    if (tid == 0 && rank == 0) atomicOr(&g_status_topk, kDevBadPos);
    qp = -1;  // no valid history: all -1
  }
  const int n = qp + 1;
  const int K = a.K;
  int32_t* out = a.idx + static_cast<int64_t>(t) * K;
  if (n <= K) {  // cluster-uniform
    for (int i = rank * kThreads + tid; i < K; i += CL * kThreads) out[i] = (i < n) ? i : -1;
    return;
  }
  // this CTA's slice [lo, hi) of the history (slice starts are multiples of 4)
  const int slice = ((n + CL - 1) / CL + 3) & ~3;
  const int lo = min(n, rank * slice), hi = min(n, lo + slice);
  const int len = hi - lo;
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld + lo;
  const bool cached = slice <= a.cache_keys;
  auto key_at = [&](int i) -> uint32_t { return cached ? keys_s[i] : order_key(__ldg(row + i)); };

  if (cached) {
    // scores -> keys in shared memory: 16-byte loads, several in flight per thread
    const int n4 = len >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldg(row4 + i);
      reinterpret_cast<uint4*>(keys_s)[i] =
          make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
    }
    for (int i = 4 * n4 + tid; i < len; i += kThreads) keys_s[i] = order_key(__ldg(row + i));
  }

  // Warp w owns slice positions [w*wl, w*wl + wl) (wl a multiple of 128) in both
  // the digit passes and the compaction, so its per-warp histograms also give it
  // the counts the compaction needs: keys above the threshold and keys equal to it.
  const int warp = tid >> 5;
  const int wl = ((len + kWarps - 1) / kWarps + 127) & ~127;
  const int wlo = min(len, warp * wl), whi = min(len, wlo + wl);
  uint32_t n_gt = 0, n_eq = 0;
  uint32_t prefix = 0, pmask = 0;
  if (tid == 0) {
    s_gt_before = 0;
    s_eq_before = 0;
  }
  uint32_t rem = static_cast<uint32_t>(K);  // how many of the keys matching `prefix` to keep
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    // this buffer was last read by the cluster two passes ago, before the
    // barrier of the previous pass
    uint32_t* hist = hist2[pass & 1];
    {
      uint32_t* wflat = &whist[0][0];
      for (int i = tid; i < kWarps * 256; i += kThreads) wflat[i] = 0;
    }
    __syncthreads();
    {
      uint32_t* wh = whist[warp];
      auto count = [&](uint32_t k) {
        if ((k & pmask) == prefix) atomicAdd(&wh[(k >> shift) & 255u], 1u);
      };
      for (int b = wlo; b < whi; b += 128) {
        const int i4 = b + 4 * lane;   // this lane's four consecutive keys
        if (i4 + 3 < whi) {
          uint4 k4;
          if (cached) {
            k4 = reinterpret_cast<const uint4*>(keys_s)[i4 >> 2];
          } else {
            const float4 v = __ldg(reinterpret_cast<const float4*>(row + i4));
            k4 = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
          }
          count(k4.x);
          count(k4.y);
          count(k4.z);
          count(k4.w);
        } else {
          for (int e = 0; e < 4; ++e)
            if (i4 + e < whi) count(key_at(i4 + e));
        }
      }
    }
    __syncthreads();
    for (int b = tid; b < 256; b += kThreads) {
      uint32_t v = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += whist[w][b];
      hist[b] = v;
    }
    cluster.sync();  // every slice's histogram complete
    // thread i < 256 reads bin i of every slice (all ranks' loads in flight at
    // once), keeping the sum over the slices before this one for later
    uint32_t before_i = 0;
    if (tid < 256) {
      uint32_t part[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) part[r] = r < CL ? cluster.map_shared_rank(hist, r)[tid] : 0u;
      uint32_t v = 0;
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r) {
        v += part[r];
        before_i += r < rank ? part[r] : 0u;
      }
      ghist[tid] = v;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending); find the digit where
      // the count of larger-or-equal digits first reaches `rem`.
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = ghist[255 - (8 * lane + j)];
        loc += c[j];
      }
      uint32_t inc = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      uint32_t run = inc - loc;
      if (run < rem && inc >= rem) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < rem && run + c[j] >= rem) {
            s_digit = 255u - (8u * lane + j);
            s_rem = rem - run;
            s_bucket = c[j];
          }
          run += c[j];
        }
      }
    }
    __syncthreads();  // s_* visible in this CTA
    {
      // this warp's keys above the chosen digit (above the threshold for good)
      // and on it (equal to the threshold so far)
      const uint32_t d = s_digit;
      uint32_t above = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t bin = 8u * lane + j;
        above += bin > d ? whist[warp][bin] : 0u;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
      n_gt += above;
      n_eq = whist[warp][d];
      // the earlier slices' keys above the chosen digit, and on it
      if (tid < 256) {
        uint32_t bg = tid > static_cast<int>(d) ? before_i : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bg += __shfl_xor_sync(0xffffffffu, bg, o);
        if (lane == 0 && bg) atomicAdd(&s_gt_before, bg);
        if (tid == static_cast<int>(d)) s_eq_before = before_i;
      }
    }
    prefix |= s_digit << shift;
    pmask |= 255u << shift;
    rem = s_rem;
    const bool whole = (s_bucket == rem);
    __syncthreads();  // s_* and the per-warp histograms are rewritten next pass
    if (whole) break;  // cluster-uniform (same histogram everywhere)
  }

  // The last distributed read of the peers' histograms is done: signal that,
  // and wait for the others only before exit.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // Ordered compaction over the same warp ranges.  The
  // slices before this one hold eq_before keys equal to the threshold (the first
  // ones in position order, so min(eq_before, rem) of them are selected) and
  // gt_before keys above it.
  const uint32_t lt_mask = (1u << lane) - 1u;
  uint32_t eq_w, gt_w;
  warp_offsets2(n_eq, n_gt, scan_buf, &eq_w, &gt_w);
  const uint32_t eq_before = s_eq_before;
  const uint32_t sel_before = s_gt_before + min(eq_before, rem);
  // this warp's first equal-key rank and first output slot
  uint32_t eq_rank = eq_before + eq_w;
  uint32_t pos = sel_before + gt_w + (eq_before >= rem ? 0u : min(eq_w, rem - eq_before));
  // 128 positions per step, four consecutive ones per lane (lane-major order);
  // one ballot per sub-position gives every lane the counts before its keys
  for (int b = wlo; b < whi; b += 128) {
    const int i4 = b + 4 * lane;
    uint32_t k[4];
    if (cached && i4 + 3 < whi) {
      const uint4 k4 = reinterpret_cast<const uint4*>(keys_s)[i4 >> 2];
      k[0] = k4.x;
      k[1] = k4.y;
      k[2] = k4.z;
      k[3] = k4.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = i4 + e < whi ? key_at(i4 + e) : 0u;
    }
    uint32_t eqb = 0, gtb = 0;   // bit e: key i4 + e equal to / above the threshold
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t km = k[e] & pmask;
      const bool valid = i4 + e < whi;
      eqb |= (valid && km == prefix) ? (1u << e) : 0u;
      gtb |= (valid && km > prefix) ? (1u << e) : 0u;
    }
    uint32_t eq_before_lane = 0, eq_total = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = __ballot_sync(0xffffffffu, (eqb >> e) & 1u);
      eq_before_lane += __popc(m & lt_mask);
      eq_total += __popc(m);
    }
    uint32_t selb = gtb, r = eq_rank + eq_before_lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((eqb >> e) & 1u) {
        if (r < rem) selb |= 1u << e;
        ++r;
      }
    }
    uint32_t sel_before_lane = 0, sel_total = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = __ballot_sync(0xffffffffu, (selb >> e) & 1u);
      sel_before_lane += __popc(m & lt_mask);
      sel_total += __popc(m);
    }
    uint32_t o = pos + sel_before_lane;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((selb >> e) & 1u) out[o++] = lo + i4 + e;
    }
    eq_rank += eq_total;
    pos += sel_total;
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // peers may still read this histogram
}

}  // namespace

cudaError_t launch_topk(const SeqArgs& seq, const float* scores, int64_t ld, int32_t K,
                        int32_t* idx, const LaunchEnv& env, std::string* plan) {
  if (seq.T == 0) {
    *plan += "topk[empty]";
    return cudaSuccess;
  }
  // As many CTAs as fit the GPU in one wave (a small batch splits each history
  // over a cluster), no more than the history can feed, and enough to keep a
  // slice within the shared-memory key cache when the cluster can.
  const int want = std::max(1, env.num_sms / seq.T);   // one wave: T x cluster <= SMs
  const int feed = std::max(1, seq.max_ctx / kMinSliceKeys);
  const int fit = (seq.max_ctx + kCacheKeys - 1) / kCacheKeys;
  const int cl = std::max(1, std::min(kMaxCluster, std::max(std::min(want, feed), fit)));
  const int slice = ((seq.max_ctx + cl - 1) / cl + 3) & ~3;
  const bool cached = slice <= kCacheKeys;
  const size_t smem = cached ? static_cast<size_t>(slice) * 4 : 0;
  const cudaError_t attr_err =
      ensure_smem_limit(reinterpret_cast<const void*>(topk_kernel), kCacheKeys * 4, env.device);
  if (attr_err != cudaSuccess) return attr_err;
  TopkArgs a{scores, ld, seq.q_pos, seq.max_ctx, K, idx, cached ? slice : 0, seq.T};
  cudaError_t e = launch_kernel(topk_kernel, dim3(seq.T * cl), dim3(kThreads), smem, env.stream, /*pdl=*/false, cl, a);
  char buf[96];
  snprintf(buf, sizeof(buf), "topk_radix[cluster=%d,%s]", cl, cached ? "smem" : "global");
  *plan += buf;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dsa
