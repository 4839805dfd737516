// Per-query Top-K over the causal history (step 2 of the DSA path).
//
// "Large Language Model Inference Acceleration in Practice", section 1.2: the
// lightning indexer selects the Top-K most relevant historical positions for the
// current query.  For query t with history n = q_pos[t] + 1 the kernel returns
// the min(K, n) positions with the largest fp32 scores, ties to the lower
// position, as an ascending list followed by -1 padding.
//
// Stand-alone kernel over a score matrix in global memory: a query's history is
// split into contiguous slices over the CTAs of a thread-block cluster (1 to 16
// CTAs of 512 threads, as many as fit the GPU in one wave), each slice's scores
// turned into order-preserving keys in that CTA's shared memory while its first
// histogram is counted, then the cluster radix select of topk_select.cuh.
#include <algorithm>
#include <cstdio>

#include "dsa_device.cuh"
#include "dsa_internal.h"
#include "topk_select.cuh"

DSA_DEFINE_STATUS_WORD(topk)

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxCluster = 8;          // portable cluster size
constexpr int kMaxClusterOne = 16;      // non-portable, for a single query
constexpr int kMinSliceKeys = 1024;     // smallest history slice worth a CTA
constexpr int kCacheKeys = 48 * 1024;   // shared-memory key cache per CTA (192 KB)

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

__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
  grid_dep_wait();
  // The attention kernel that follows may start now: it stages its query and
  // waits for this grid before it reads the indices.
  grid_dep_launch();
  extern __shared__ uint32_t keys_s[];
  __shared__ SelectSmem sel;
  const int CL = static_cast<int>(cl_size());
  const int rank = static_cast<int>(cl_rank());
  // clusters take queries last-first: with causal histories (prefill) the longest
  // histories start first and the short ones fill the tail of the launch
  const int t = a.T - 1 - static_cast<int>(blockIdx.x) / CL;
  const int tid = threadIdx.x;
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
  select_prepare<kThreads>(&sel, CL);
  // this CTA's slice [lo, hi) of the history (slice starts are multiples of 4)
  const int slice = ((n + CL - 1) / CL + 3) & ~3;
  const int lo = min(n, rank * slice), hi = min(n, lo + slice);
  const int len = hi - lo;
  const float* row = a.scores + static_cast<int64_t>(t) * a.ld + lo;
  const bool cached = slice <= a.cache_keys;
  if (cached) {
    // scores -> keys in shared memory (16-byte loads, several in flight per
    // thread), counted into the first histogram on the way
    const int n4 = len >> 2;
    const float4* row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldg(row4 + i);
      const uint4 k = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
      reinterpret_cast<uint4*>(keys_s)[i] = k;
      select_count0(&sel, k.x);
      select_count0(&sel, k.y);
      select_count0(&sel, k.z);
      select_count0(&sel, k.w);
    }
    for (int i = 4 * n4 + tid; i < len; i += kThreads) {
      const uint32_t k = order_key(__ldg(row + i));
      keys_s[i] = k;
      select_count0(&sel, k);
    }
    select_run<kThreads>(
        &sel, [&](int i) -> uint32_t { return keys_s[i]; },
        [&](int i) -> uint4 { return reinterpret_cast<const uint4*>(keys_s)[i >> 2]; }, len, lo, K, out, true);
  } else {
    // slice starts are multiples of 4: 16-byte loads of 4 scores
    select_run<kThreads>(
        &sel, [&](int i) -> uint32_t { return order_key(__ldg(row + i)); },
        [&](int i) -> uint4 {
          const float4 v = __ldg(reinterpret_cast<const float4*>(row + i));
          return make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        },
        len, lo, K, out, false);
  }
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
  const cudaError_t attr_err =
      ensure_smem_limit(reinterpret_cast<const void*>(topk_kernel), kCacheKeys * 4, env.device);
  if (attr_err != cudaSuccess) return attr_err;
  // A single query may take a non-portable cluster of 16 CTAs when the GPU can
  // place one (decode batch 1: 0.15 us per step faster than 8 in an A/B; with
  // four queries 16 was slower, the clusters crowding the attention launched
  // behind them)
  int max_cl = kMaxCluster;
  if (seq.T == 1 && std::min(want, feed) > kMaxCluster &&
      cluster_fits(reinterpret_cast<const void*>(topk_kernel), env.device, kMaxClusterOne, kThreads, kCacheKeys * 4))
    max_cl = kMaxClusterOne;
  const int cl = std::max(1, std::min(max_cl, std::max(std::min(want, feed), fit)));
  const int slice = ((seq.max_ctx + cl - 1) / cl + 3) & ~3;
  const bool cached = slice <= kCacheKeys;
  const size_t smem = cached ? static_cast<size_t>(slice) * 4 : 0;
  TopkArgs a{scores, ld, seq.q_pos, seq.max_ctx, K, idx, cached ? slice : 0, seq.T};
  // Programmatic dependent launch: the clusters are placed as the indexer's CTAs
  // finish (each triggers its dependents when its tiles are done) and wait for
  // the scores in griddepcontrol.wait, instead of launching after the indexer's
  // grid has drained (decode batch 1: 0.6 us per step, long-context batch 4:
  // 0.7 us).
  cudaError_t e = launch_kernel(topk_kernel, dim3(seq.T * cl), dim3(kThreads), smem, env.stream, /*pdl=*/true, cl, a);
  char buf[96];
  snprintf(buf, sizeof(buf), "topk_radix[cluster=%d,%s]", cl, cached ? "smem" : "global");
  *plan += buf;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dsa
