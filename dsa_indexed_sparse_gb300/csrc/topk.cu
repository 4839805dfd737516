// Per-query Top-K over the causal history (step 2 of the DSA path).
//
// "Large Language Model Inference Acceleration in Practice", section 1.2: the
// lightning indexer selects the Top-K most relevant historical positions for the
// current query.  For query t with history n = q_pos[t] + 1 the kernel returns
// the min(K, n) positions with the largest fp32 scores, ties to the lower
// position, as an ascending list followed by -1 padding.
//
// Exact radix select, one CTA (1024 threads) per query:
//  * scores -> order-preserving uint32 keys (-0.0 folded onto +0.0);
//  * up to four 8-bit digit passes, each a shared-memory histogram of the keys
//    that still match the selected prefix, narrow the K-th largest key; a pass
//    stops early when the bucket holding the K-th key is taken whole;
//  * an ordered compaction (contiguous per-thread chunks, two block scans) keeps
//    every key above the threshold and the first `remaining` keys equal to it,
//    which writes the output already sorted.
// Keys are cached in shared memory when the history fits (<= 48K positions);
// longer histories re-read the scores from global memory (L2) on every pass.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

DSA_DEFINE_STATUS_WORD(topk)

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheKeys = 48 * 1024;  // 192 KB of shared memory

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
  int32_t cache_keys;  // keys cached in dynamic smem (0 = none)
};

// Exclusive scan of one value per warp; every thread gets (its warp's offset,
// block total).  Uses `buf` [kWarps] and two __syncthreads.
__device__ __forceinline__ void warp_offsets(uint32_t warp_count, uint32_t* buf, uint32_t* excl,
                                             uint32_t* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) buf[warp] = warp_count;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = buf[lane];
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    buf[lane] = inc - v;                       // exclusive
    if (lane == 31) buf[kWarps] = inc;         // total
  }
  __syncthreads();
  *excl = buf[warp];
  *total = buf[kWarps];
}

// Exclusive block-wide scan of one value per thread (all kThreads threads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* buf, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  uint32_t w_excl, tot;
  warp_offsets(__shfl_sync(0xffffffffu, inc, 31), buf, &w_excl, &tot);
  *total = tot;
  return w_excl + inc - v;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
  extern __shared__ uint32_t keys_s[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scan_buf[kWarps + 1];
  __shared__ uint32_t s_digit, s_rem, s_bucket;

  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  int qp = __ldg(a.q_pos + t);
  if (qp < 0 || qp >= a.max_ctx) {
    if (tid == 0) atomicOr(&g_status_topk, kDevBadPos);
    qp = -1;  // no valid history: all -1
  }
  const int n = qp + 1;
  const int K = a.K;
  int32_t* out = a.idx + static_cast<int64_t>(t) * K;
  if (n <= K) {
    for (int i = tid; i < K; i += kThreads) out[i] = (i < n) ? i : -1;
    return;
  }
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld;
  const bool cached = n <= a.cache_keys;
  auto key_at = [&](int i) -> uint32_t { return cached ? keys_s[i] : order_key(__ldg(row + i)); };

  if (cached) {
    // scores -> keys in shared memory: 16-byte loads, several in flight per thread
    const int n4 = n >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldg(row4 + i);
      reinterpret_cast<uint4*>(keys_s)[i] =
          make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
    }
    for (int i = 4 * n4 + tid; i < n; i += kThreads) keys_s[i] = order_key(__ldg(row + i));
    __syncthreads();
  }

  uint32_t prefix = 0, pmask = 0;
  uint32_t rem = static_cast<uint32_t>(K);  // how many of the keys matching `prefix` to keep
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    // Scores cluster in few top-digit buckets: lanes hitting the same bucket
    // combine their counts (match_any) so each bucket takes one atomic per warp.
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + tid;
      bool act = false;
      uint32_t k = 0;
      if (i < n) {
        k = key_at(i);
        act = (k & pmask) == prefix;
      }
      const uint32_t active = __ballot_sync(0xffffffffu, act);
      if (act) {
        const uint32_t bin = (k >> shift) & 255u;
        const uint32_t peers = __match_any_sync(active, bin);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending); find the digit where
      // the count of larger-or-equal digits first reaches `rem`.
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - (8 * lane + j)];
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
    __syncthreads();
    prefix |= s_digit << shift;
    pmask |= 255u << shift;
    rem = s_rem;
    const bool whole = (s_bucket == rem);
    __syncthreads();  // s_* are rewritten next pass
    if (whole) break;
  }

  // Ordered compaction.  Thread `tid` owns positions [tid*c, tid*c + c), c odd
  // (so the shared-memory reads of a warp fall in distinct banks).  Keep every
  // key above the threshold and, in position order, the first `rem` keys equal
  // to it; the output comes out in ascending position order.
  int c = (n + kThreads - 1) / kThreads;
  c |= 1;
  const int lo = min(n, tid * c), hi = min(n, lo + c);
  uint32_t n_eq = 0;
  for (int i = lo; i < hi; ++i) n_eq += (key_at(i) & pmask) == prefix;
  uint32_t tot;
  uint32_t eq_rank = block_excl_scan(n_eq, scan_buf, &tot);
  __syncthreads();
  uint32_t n_sel = 0;
  {
    uint32_t r = eq_rank;
    for (int i = lo; i < hi; ++i) {
      const uint32_t km = key_at(i) & pmask;
      if (km > prefix) {
        ++n_sel;
      } else if (km == prefix) {
        n_sel += r < rem;
        ++r;
      }
    }
  }
  uint32_t pos = block_excl_scan(n_sel, scan_buf, &tot);
  for (int i = lo; i < hi && n_sel > 0; ++i) {
    const uint32_t km = key_at(i) & pmask;
    bool sel = km > prefix;
    if (km == prefix) {
      sel = eq_rank < rem;
      ++eq_rank;
    }
    if (sel) {
      out[pos++] = i;
      --n_sel;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const SeqArgs& seq, const float* scores, int64_t ld, int32_t K,
                        int32_t* idx, const LaunchEnv& env, std::string* plan) {
  if (seq.T == 0) {
    *plan += "topk[empty]";
    return cudaSuccess;
  }
  const int cache = std::min(seq.max_ctx, kCacheKeys);
  const size_t smem = (seq.max_ctx <= kCacheKeys) ? static_cast<size_t>(cache) * 4 : 0;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kCacheKeys * 4);
  });
  if (attr_err != cudaSuccess) return attr_err;
  TopkArgs a{scores, ld, seq.q_pos, seq.max_ctx, K, idx, smem ? cache : 0};
  topk_kernel<<<seq.T, kThreads, smem, env.stream>>>(a);
  char buf[96];
  snprintf(buf, sizeof(buf), "topk_radix[%s]", smem ? "smem" : "global");
  *plan += buf;
  return cudaGetLastError();
}

}  // namespace dsa
