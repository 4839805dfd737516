// Exact Top-K selection over one query's history, split into contiguous slices
// held in the shared memory of the CTAs of a thread-block cluster (step 2 of the
// DSA path: "Large Language Model Inference Acceleration in Practice", section
// 1.2 -- the K positions with the largest index scores, ties to the lower
// position).  Used by the stand-alone Top-K kernel and by the fused decode
// kernel, whose indexer epilogue writes the keys straight into shared memory.
//
// Keys are order-preserving uint32 images of the fp32 scores (-0.0 folded onto
// +0.0).  Radix select over at most three digits, bits [31:21], [20:10], [9:0]
// (11 + 11 + 10): the first digit is sign, exponent and two mantissa bits, so
// after the second the boundary bin is 2^-13 of an octave wide and usually
// holds the K-th key alone -- two passes.  A pass:
//   * every CTA builds the histogram of the keys of its slice that match the
//     digits chosen so far (shared-memory atomics);
//   * it pushes each non-empty bin into the same bin of EVERY CTA of the
//     cluster (red.shared::cluster.add), so after one cluster barrier each CTA
//     holds the cluster's histogram locally and picks the same digit by itself
//     -- no remote reads;
//   * the histograms alternate between two buffers: the one for the next pass is
//     zeroed by its owner before it arrives at this pass's barrier, i.e. before
//     any peer can push into it.
// Compaction: each CTA counts, per warp, its keys above the threshold and equal
// to it; the CTA totals go to the higher-ranked CTAs (one more barrier); keys
// above are all taken, equal keys in position order up to the remaining count,
// written in ascending position order (ballots over 32 consecutive keys give
// every lane its slot).
#pragma once

#include "dsa_device.cuh"

namespace dsa {

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;  // -0.0 == +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------- cluster PTX
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cl_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cl_map(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cl_red_add(uint32_t cl_addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_store(uint32_t cl_addr, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}
// Every thread of every CTA of the cluster arrives / waits (warp-converged).
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

constexpr int kSelBins = 2048;
constexpr int kSelMaxCluster = 16;

struct alignas(16) SelectSmem {
  uint32_t bins[2][kSelBins];        // the cluster's histogram, by pass parity (peers push into it)
  uint32_t local[kSelBins];          // this CTA's histogram of the current pass
  uint32_t wred[2][32];              // per-warp partials of the block scans
  uint32_t cnt[kSelMaxCluster][2];   // (above, equal) counts of the lower ranks' slices
  uint32_t digit, rem, bucket;
};

__device__ __forceinline__ int sel_shift(int pass) { return pass == 0 ? 21 : (pass == 1 ? 10 : 0); }
__device__ __forceinline__ uint32_t sel_mask(int pass) { return pass == 2 ? 1023u : 2047u; }

// Zeroes the histograms and arrives at the cluster barrier that select_run's
// first wait completes: no peer pushes into this CTA's histogram before it is
// zeroed.  Every thread of the CTA calls it (and then select_run).
template <int kThreads>
__device__ __forceinline__ void select_prepare(SelectSmem* sm, int CL) {
  for (int i = threadIdx.x; i < 3 * kSelBins; i += kThreads) (&sm->bins[0][0])[i] = 0u;
  __syncthreads();
  if (CL > 1) cl_arrive();
}

// Adds this thread's share of the keys to the pass-0 histogram (callers that
// produce keys themselves do this as they write them; select_run does it
// otherwise).
__device__ __forceinline__ void select_count0(SelectSmem* sm, uint32_t key) {
  atomicAdd(&sm->local[key >> 21], 1u);
}

// Block-wide exclusive scan over threads of two values, plus the totals: warp
// scans, then one warp scans the warp totals (two barriers).
template <int kThreads>
__device__ __forceinline__ void block_excl2(uint32_t a, uint32_t b, uint32_t (*wred)[32], uint32_t* ea,
                                            uint32_t* eb, uint32_t* ta, uint32_t* tb) {
  constexpr int kWarps = kThreads / 32;
  static_assert(kWarps <= 31, "one slot per warp plus the total");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t ua = __shfl_up_sync(0xffffffffu, ia, o), ub = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += ua;
      ib += ub;
    }
  }
  if (lane == 31) {
    wred[0][warp] = ia;
    wred[1][warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t va = lane < kWarps ? wred[0][lane] : 0u, vb = lane < kWarps ? wred[1][lane] : 0u;
    uint32_t xa = va, xb = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ua = __shfl_up_sync(0xffffffffu, xa, o), ub = __shfl_up_sync(0xffffffffu, xb, o);
      if (lane >= o) {
        xa += ua;
        xb += ub;
      }
    }
    // exclusive prefixes in [0, kWarps), totals in slot 31
    if (lane < kWarps) {
      wred[0][lane] = xa - va;
      wred[1][lane] = xb - vb;
    }
    if (lane == 31) {
      wred[0][31] = xa;
      wred[1][31] = xb;
    }
  }
  __syncthreads();
  *ea = wred[0][warp] + ia - a;
  *eb = wred[1][warp] + ib - b;
  *ta = wred[0][31];
  *tb = wred[1][31];
}

// Pushes this CTA's histogram bins [0, nbins) into bin b of `hist` in every CTA
// of the cluster, and clears them locally.  Bins are strided over the threads
// (the non-empty ones are few and adjacent, so each lands on its own thread).
template <int kThreads>
__device__ __forceinline__ void push_bins(uint32_t* local, uint32_t* hist, int nbins, int CL) {
  for (int b = threadIdx.x; b < nbins; b += kThreads) {
    const uint32_t v = local[b];
    if (v) {
      local[b] = 0u;
      const uint32_t a = smem_u32(hist + b);
      for (int r = 0; r < CL; ++r) cl_red_add(cl_map(a, static_cast<uint32_t>(r)), v);
    }
  }
}

// Selects, over the cluster, the min(K, n) largest keys of positions [0, n) of
// one query (n > K), this CTA holding positions [lo, lo + len) through
// key_at(i), i in [0, len); writes the selected positions in ascending order to
// out[0, K) (n > K: exactly K of them).  The pass-0 histogram of this CTA's keys
// must already be in sm->local when have_local0; select_prepare must have run.
template <int kThreads, typename KeyAt, typename Key4At>
__device__ void select_run(SelectSmem* sm, KeyAt key_at, Key4At key4_at, int len, int lo, int K, int32_t* out,
                           bool have_local0) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kPer = (kSelBins + kThreads - 1) / kThreads;   // bins per thread in the digit scan
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int CL = static_cast<int>(cl_size());
  const uint32_t rank = cl_rank();
  if (!have_local0) {
    for (int i = tid; i < len; i += kThreads) select_count0(sm, key_at(i));
  }
  __syncthreads();
  if (CL > 1) cl_wait();   // every CTA's histograms are zeroed (select_prepare)

  uint32_t prefix = 0, pmask = 0, rem = static_cast<uint32_t>(K);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = sel_shift(pass);
    const uint32_t mask = sel_mask(pass);
    if (pass > 0) {
      // keys four at a time (the slice starts on a 16-byte boundary), then the tail
      const int len4 = len & ~3;
      for (int i = 4 * tid; i < len4; i += 4 * kThreads) {
        const uint4 k4 = key4_at(i);
        const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((kk[e] & pmask) == prefix) atomicAdd(&sm->local[(kk[e] >> shift) & mask], 1u);
      }
      for (int i = len4 + tid; i < len; i += kThreads) {
        const uint32_t k = key_at(i);
        if ((k & pmask) == prefix) atomicAdd(&sm->local[(k >> shift) & mask], 1u);
      }
      __syncthreads();
    }
    uint32_t* hist = sm->bins[pass & 1];
    if (CL > 1) {
      // push the non-empty bins into every CTA's copy (this one's included)
      push_bins<kThreads>(sm->local, hist, static_cast<int>(mask) + 1, CL);
      // the buffer of the next pass: last read by this CTA's scan of the previous
      // pass; peers push into it only after this pass's barrier
      if (pass >= 1 && pass < 2)
        for (int b = tid; b < kSelBins; b += kThreads) sm->bins[(pass + 1) & 1][b] = 0u;
      cl_arrive();
      cl_wait();
    } else {
      // one CTA: its histogram is the query's (bins beyond this pass's digit range
      // cleared: the buffer held an earlier pass)
      for (int b = tid; b < kSelBins; b += kThreads) {
        hist[b] = b <= static_cast<int>(mask) ? sm->local[b] : 0u;
        sm->local[b] = 0u;
      }
      __syncthreads();
    }
    // the bin holding the rem-th largest key: thread i owns kPer consecutive bins
    // in descending order
    uint32_t c[kPer], s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int bin = kSelBins - 1 - (tid * kPer + j);
      c[j] = bin >= 0 ? hist[bin] : 0u;
      s += c[j];
    }
    uint32_t excl, dummy, tot, dtot;
    block_excl2<kThreads>(s, 0u, sm->wred, &excl, &dummy, &tot, &dtot);
    if (excl < rem && excl + s >= rem) {
      uint32_t run = excl;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        if (run < rem && run + c[j] >= rem) {
          sm->digit = static_cast<uint32_t>(kSelBins - 1 - (tid * kPer + j));
          sm->rem = rem - run;
          sm->bucket = c[j];
        }
        run += c[j];
      }
    }
    __syncthreads();
    const uint32_t d = sm->digit;
    prefix |= d << shift;
    pmask |= mask << shift;
    rem = sm->rem;
    const bool whole = sm->bucket == rem;
    // (the pass-1 buffer was zeroed before the pass-0 barrier by select_prepare;
    // bins[0] for pass 2 by the code above in pass 1)
    if (whole) break;   // uniform: the same histogram in every CTA
  }

  // ---- compaction: keys above the threshold, and the first `rem` (cluster-wide,
  // by position) equal to it.  Warp w owns slice positions [w*wl, w*wl + wl).
  const int wl = ((len + kWarps - 1) / kWarps + 127) & ~127;
  const int wlo = min(len, warp * wl), whi = min(len, wlo + wl);
  uint32_t n_gt = 0, n_eq = 0;
  for (int b = wlo; b < whi; b += 128) {   // 128 keys a step, four per lane
    const int i4 = b + 4 * lane;
    uint32_t k[4];
    if (i4 + 3 < whi) {
      const uint4 v = key4_at(i4);
      k[0] = v.x;
      k[1] = v.y;
      k[2] = v.z;
      k[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = i4 + e < whi ? key_at(i4 + e) : 0u;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i4 + e < whi) {
        const uint32_t km = k[e] & pmask;
        n_gt += km > prefix ? 1u : 0u;
        n_eq += km == prefix ? 1u : 0u;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o);
    n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o);
  }
  // warp offsets: lane 0 of each warp contributes its warp's counts
  uint32_t gt_w, eq_w, gt_cta, eq_cta;
  block_excl2<kThreads>(lane == 0 ? n_gt : 0u, lane == 0 ? n_eq : 0u, sm->wred, &gt_w, &eq_w, &gt_cta, &eq_cta);
  gt_w = __shfl_sync(0xffffffffu, gt_w, 0);
  eq_w = __shfl_sync(0xffffffffu, eq_w, 0);
  uint32_t gt_before = 0, eq_before = 0;
  if (CL > 1) {
    if (tid < CL && tid > static_cast<int>(rank)) {
      cl_store(cl_map(smem_u32(&sm->cnt[rank][0]), static_cast<uint32_t>(tid)), gt_cta);
      cl_store(cl_map(smem_u32(&sm->cnt[rank][1]), static_cast<uint32_t>(tid)), eq_cta);
    }
    cl_arrive();
    cl_wait();
    for (int r = 0; r < static_cast<int>(rank); ++r) {
      gt_before += sm->cnt[r][0];
      eq_before += sm->cnt[r][1];
    }
  }
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t sel_before = gt_before + min(eq_before, rem);
  uint32_t eq_rank = eq_before + eq_w;   // cluster-wide rank of this warp's first equal key
  uint32_t pos = sel_before + gt_w + (eq_before >= rem ? 0u : min(eq_w, rem - eq_before));
  for (int b = wlo; b < whi; b += 128) {
    const int i4 = b + 4 * lane;
    uint32_t eqb = 0, gtb = 0;   // bit e: key i4 + e equal to / above the threshold
    uint32_t k[4];
    if (i4 + 3 < whi) {
      const uint4 v = key4_at(i4);
      k[0] = v.x;
      k[1] = v.y;
      k[2] = v.z;
      k[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) k[e] = i4 + e < whi ? key_at(i4 + e) : 0u;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i4 + e < whi) {
        const uint32_t km = k[e] & pmask;
        eqb |= km == prefix ? (1u << e) : 0u;
        gtb |= km > prefix ? (1u << e) : 0u;
      }
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
}

}  // namespace dsa
