// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA tile loads, tcgen05 (UMMA) descriptors / MMA / TMEM access,
// cp.async and FP8 conversion.  Inline PTX only; no library kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

// Device status flags (sticky, OR-ed into a per-translation-unit word).
enum : uint32_t {
  kDevTimeout = 1u,     // a pipeline wait gave up
  kDevBadIndex = 2u,    // page id / selected index out of range
  kDevBadPos = 4u,      // q_pos < 0 or q_pos >= max_ctx
  kDevBadGroup = 8u,    // q_per_seq promise broken (group spans two sequences)
  kDevConfig = 16u,     // a launch configuration the kernel cannot run (e.g. its
                        // re-aligned shared-memory layout does not fit); nothing done
};

// Upper bound of any single pipeline wait (the longest legitimate wait is a few
// microseconds; a stuck pipeline gives up after this and flags kDevTimeout).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep until the phase completes (or hint_ns
// passes): a waiting warp then takes no issue slots from the warps it shares a
// sub-partition with.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t addr, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns (or as soon as another thread of the CTA has given up), sets
// kDevTimeout in *status and returns false; never traps.  With sleep_ns > 0
// the waiting thread sleeps between polls (up to sleep_ns, woken when the
// phase completes).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          volatile int* abort_flag, uint64_t limit_ns = kWaitLimitNs,
                                          uint32_t sleep_ns = 0) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (sleep_ns ? mbar_try_wait_sleep(addr, parity, sleep_ns) : mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        atomicOr(status, kDevTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Waits for a phase without looking at the CTA's abort flag: used on the way
// out, to let asynchronous copies and tensor-core work that were issued before
// an abort finish before their shared memory or TMEM is released.  Bounded by
// limit_ns as well; returns false (and sets kDevTimeout) if it gave up.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, uint32_t* status,
                                           uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

// One lane of a converged warp (the whole warp must execute this).  tcgen05.mma
// issued from a converged warp through elect.sync costs ~40-65 cycles per
// instruction on sm_103a; issued from a lone lane of a diverged warp ~100-130.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------- proxies / fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// 2-D tiled load, completion counted in bytes on `bar`.  c0 = innermost coordinate
// (elements), c1 = row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* map, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}



// Programmatic dependent launch.  grid_dep_wait blocks until every grid this
// launch depends on has completed and its writes are visible (at once when the
// kernel was launched without programmatic stream serialization); nothing that
// an earlier kernel may write -- inputs included -- is read before it.
// grid_dep_launch lets the next kernel on the stream launch now, so that its
// launch and set-up overlap this grid's tail.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Asks L2 to fetch the line holding addr (no data returned to the SM).
__device__ __forceinline__ void prefetch_l2(const void* addr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(addr));
}

// ---------------------------------------------------------------- cp.async (16 B)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrives on the mbarrier once all of this thread's earlier cp.async copies have
// landed (the arrival is counted in the barrier's expected count: .noinc).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Stores 32 rows of 128 bytes, held one row per lane (v = the row's 32 words), to
// global memory (row r at dst + r * stride_bytes) as whole 128-byte lines: the
// warp transposes through a 4 KB staging buffer at stg (XOR-swizzled 16-byte
// slots, conflict-free both ways).  Without it every store instruction would
// scatter 16 bytes to each of 32 rows.
__device__ __forceinline__ void warp_store_rows128(uint32_t stg, const uint32_t (&v)[32], uint8_t* dst,
                                                   int64_t stride_bytes, int lane) {
#pragma unroll
  for (int k = 0; k < 8; ++k)
    st_shared_v4(stg + lane * 128 + ((k ^ (lane & 7)) << 4), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = i * 4 + (lane >> 3), c4 = lane & 7;
    const uint4 w = ld_shared_v4(stg + row * 128 + ((c4 ^ (row & 7)) << 4));
    *reinterpret_cast<uint4*>(dst + row * stride_bytes + c4 * 16) = w;
  }
  __syncwarp();
}
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------- tcgen05 / TMEM
// Warp-wide: allocates `ncols` TMEM columns (power of two >= 32) and writes the
// base address to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16/f16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, bf16/f16 inputs: A (M=128 rows) is read from
// tensor memory, row m in lane m, 2 consecutive K elements per 32-bit column.
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same for 8-bit float inputs (e4m3/e5m2), fp32 accumulate.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every previously issued tcgen05.mma of this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Instruction descriptor (kind::f16 / kind::f8f6f4): fp32 accumulator,
// a_fmt/b_fmt = 1 for bf16 (kind::f16) or 0 for e4m3 (kind::f8f6f4).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, bool a_mn_major,
                                                  bool b_mn_major, uint32_t M, uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
constexpr uint32_t kFmtBF16 = 1;
constexpr uint32_t kFmtE4M3 = 0;
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSw128 = 2;

// Shared-memory matrix descriptor.  lbo/sbo in bytes (multiples of 16).
// K-major SWIZZLE_128B: rows of 128 B, 8-row atoms 1024 B apart (sbo), lbo unused.
// MN-major SWIZZLE_128B: lbo = stride between 128-B-wide MN atoms, sbo = stride
// between groups of 8 K-rows.  No swizzle, K-major: 8x16B core matrices, lbo =
// stride between core matrices along K, sbo = along M/N.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// 32 lanes x 32 bit, 32 consecutive columns: thread i of the warp gets lane
// (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- numerics
// Two e4m3 codes (low byte first) -> two floats, exact (e4m3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}
__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v), __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}
// 2^x with the hardware approximation (PTX ex2.approx.ftz.f32; ~2 ulp, flushes
// subnormal results to zero; ex2(-inf) = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (a0, a1) += (x0 * y0, x1 * y1): two IEEE fp32 fmas (round to nearest) in one
// packed instruction (PTX fma.rn.f32x2).
__device__ __forceinline__ void fma2(float& a0, float& a1, float x0, float x1, float y0, float y1) {
  asm("{\n\t.reg .b64 ra, rx, ry;\n\t"
      "mov.b64 ra, {%0, %1};\n\tmov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
      "fma.rn.f32x2 ra, rx, ry, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
// (r0, r1) = (x0 * y0, x1 * y1): two IEEE fp32 products (round to nearest) in
// one packed instruction (PTX mul.rn.f32x2).
__device__ __forceinline__ void mul2(float& r0, float& r1, float x0, float x1, float y0, float y1) {
  asm("{\n\t.reg .b64 rx, ry, rr;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
      "mul.rn.f32x2 rr, rx, ry;\n\tmov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
// max(a, b, c) in one instruction (PTX three-input max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (r0, r1) = (x0 + y0, x1 + y1): two IEEE fp32 adds in one packed instruction
// (PTX add.rn.f32x2).
__device__ __forceinline__ void add2(float& r0, float& r1, float x0, float x1, float y0, float y1) {
  asm("{\n\t.reg .b64 rx, ry, rr;\n\t"
      "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\t"
      "add.rn.f32x2 rr, rx, ry;\n\tmov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Page-table translation: logical position s of the sequence whose table row
// starts at `bt` -> physical cache row, or -1 (and kDevBadIndex) if the page id
// is outside [0, n_pages).
__device__ __forceinline__ int64_t phys_row(const int32_t* bt, int32_t s, int32_t page_size,
                                            int64_t n_pages, uint32_t* status) {
  const int32_t page = __ldg(bt + s / page_size);
  if (page < 0 || page >= n_pages) {
    atomicOr(status, kDevBadIndex);
    return -1;
  }
  return static_cast<int64_t>(page) * page_size + (s % page_size);
}

}  // namespace dsa

// Each translation unit owns one sticky status word (device code reaches it by
// name) and exports a host-side read-and-clear helper for it.
#define DSA_DEFINE_STATUS_WORD(tag)                                        \
  static __device__ uint32_t g_status_##tag;                               \
  uint32_t dsa_status_read_clear_##tag() {                                 \
    uint32_t v = 0;                                                        \
    if (cudaMemcpyFromSymbol(&v, g_status_##tag, sizeof(v)) != cudaSuccess) \
      return 0xFFFFFFFFu;                                                  \
    const uint32_t zero = 0;                                               \
    cudaMemcpyToSymbol(g_status_##tag, &zero, sizeof(zero));               \
    return v;                                                              \
  }
