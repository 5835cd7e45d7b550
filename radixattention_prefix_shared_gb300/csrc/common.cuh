// Device helpers shared by the sm_103a kernels: bf16 unpacking, cp.async,
// mbarriers with bounded waits, and tcgen05 (TMEM + UMMA) wrappers written
// as inline PTX.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sgl_attn.h"

#define SGL_DEV __device__ __forceinline__

namespace sgl {

// ----------------------------------------------------------------- status

// Nonzero codes written into the extend workspace's status word when a
// bounded wait gives up.
enum DeviceStatus : int {
  kDevOk = 0,
  kDevWaitTimeout = 0x5701,
};

// ----------------------------------------------------------------- misc

SGL_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SGL_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 2^x for the softmax (the hardware's approximate base-2 exponential;
// exp(x) is evaluated as 2^(x * log2(e)) with log2(e) folded into the scale).
SGL_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pair arithmetic: the sm_100-family FFMA2/FADD2 instructions
// through CUDA's float2 builtins, so register pairs are allocated by the
// compiler rather than assembled with moves.
SGL_DEV float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
SGL_DEV float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
SGL_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Unpack 8 bf16 held in a uint4 into 8 floats (a bf16 is the top half of a float).
SGL_DEV void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

SGL_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

SGL_DEV uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four e4m3 codes (byte i = code i) -> two f16x2 words (codes 0,1 and 2,3)
// holding exactly code * 2^-8.  The f16 bit pattern is the code's sign at
// bit 15 and its 7 magnitude bits (exponent field e, mantissa m) at bits
// 7..13: a normal code reads as 2^(e-15) (1 + m/8) = 2^-8 * 2^(e-7) (1 + m/8),
// a subnormal one (e = 0) as the f16 subnormal m * 2^-17 = 2^-8 * m * 2^-9.
// (Codes 0x7f / 0xff, e4m3's NaN, read as +-480 * 2^-8; a saturating store
// never writes them.)
SGL_DEV void e4m3x4_to_f16x2_scaled(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t hb = ((w >> 1) & 0x3F3F3F3Fu) | (w & 0x80808080u);  // sign | bits 6..1
  const uint32_t lb = (w << 7) & 0x80808080u;                        // bit 0 -> bit 7
  lo = __byte_perm(lb, hb, 0x5140);  // (lb0, hb0, lb1, hb1)
  hi = __byte_perm(lb, hb, 0x7362);  // (lb2, hb2, lb3, hb3)
}

// ----------------------------------------------------------------- cp.async

// 16-byte global->shared copy through L2 only; src_bytes == 0 writes zeros
// without reading global memory.
SGL_DEV void cp_async_16(uint32_t dst_smem, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src),
               "r"(src_bytes)
               : "memory");
}
SGL_DEV uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
SGL_DEV void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
SGL_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SGL_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
SGL_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Arrive on `bar` once every cp.async issued so far by this thread has
// completed (the arrival is pre-counted in the barrier's expected count).
SGL_DEV void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Order generic-proxy shared-memory writes (cp.async included) that this
// thread has observed before its later async-proxy accesses (tcgen05.mma
// operand reads).
SGL_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- mbarrier

SGL_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Invalidate a barrier so that its memory can be initialised again.
SGL_DEV void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
SGL_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

SGL_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 st;\n mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// One bounded probe of the phase: the thread may sleep in hardware until the
// phase completes or about `hint_ns` elapse, so waiting warps do not spin.
SGL_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns = 100000u) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Default limit of a bounded wait (2 s of wall time).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// Wait for the phase with the given parity to complete.  Gives up after
// `limit_ns` of wall time or as soon as another thread raised *abort (when
// `abort` is given); on a timeout it raises *abort and records
// kDevWaitTimeout in *status (when given).  Returns false when it gave up.
// Limits under 100 us also shorten each probe's sleep and check the clock
// after every probe.
SGL_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int* status,
                               uint64_t limit_ns = kDefaultWaitNs) {
  const bool short_limit = limit_ns < 100000ull;
  const uint32_t hint = short_limit ? (limit_ns < 32ull ? 32u : (uint32_t)limit_ns) : 100000u;
  if (mbar_try_wait(bar, parity, hint)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if ((it & 7u) == 0 || short_limit) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        if (abort) *abort = 1;
        if (status) atomicExch(status, (int)kDevWaitTimeout);
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------- dependent launches
// A kernel launched with programmatic stream serialization may start while
// the kernel before it in the stream still runs: from the moment every CTA of
// that one has signalled (or exited).  grid_dep_wait blocks the thread until
// the kernel before has completed and its memory writes are visible; without
// such a dependency both return at once.

SGL_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
SGL_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- named barriers

SGL_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier over `nthreads` threads that also returns the OR of `pred` over them.
SGL_DEV bool bar_red_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, %3, pi;\n"
      " selp.u32 %0, 1, 0, po;\n}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

// Barrier over `nthreads` threads that returns how many of them had `pred` set.
SGL_DEV uint32_t bar_red_popc(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred pi;\n setp.ne.u32 pi, %1, 0;\n bar.red.popc.u32 %0, %2, %3, pi;\n}"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return out;
}

// ----------------------------------------------------------------- tcgen05

// TMEM allocation: one full warp executes these.
SGL_DEV void tmem_alloc(uint32_t* dst_smem_word, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem_word)),
               "r"(ncols)
               : "memory");
}
SGL_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SGL_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

SGL_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SGL_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major or MN-major operand stored in
// the 128-byte swizzled canonical layout: rows of 128 bytes (64 bf16), 16-byte
// chunk c of row r stored at chunk position c ^ (r % 8), 8-row groups of
// 1024 bytes.  lbo/sbo in bytes.
SGL_DEV uint64_t make_sw128_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version used by tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 (or, f16_ab, f16) A/B and an
// fp32 accumulator.  b_mn_major selects an MN-major (N contiguous) B operand.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major,
                                                       bool f16_ab = false) {
  return (1u << 4)                              // D format: f32
         | ((f16_ab ? 0u : 1u) << 7)            // A format: bf16 (1) or f16 (0)
         | ((f16_ab ? 0u : 1u) << 10)           // B format: same as A
         | ((b_mn_major ? 1u : 0u) << 16)       // B major-ness
         | ((uint32_t)(N >> 3) << 17)           // N / 8
         | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]
SGL_DEV void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
SGL_DEV void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
SGL_DEV void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

#define SGL_R32(a) \
  "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), \
  "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), \
  "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), \
  "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), \
  "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31])
#define SGL_W32(a) \
  "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), \
  "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]), \
  "r"(a[16]), "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]), "r"(a[21]), "r"(a[22]), \
  "r"(a[23]), "r"(a[24]), "r"(a[25]), "r"(a[26]), "r"(a[27]), "r"(a[28]), "r"(a[29]), \
  "r"(a[30]), "r"(a[31])

// Thread t of the warp reads TMEM lane (lane_base + t), columns col..col+31.
SGL_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SGL_R32(r)
      : "r"(taddr)
      : "memory");
}
SGL_DEV void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      SGL_W32(r)
      : "memory");
}
SGL_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
SGL_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
SGL_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace sgl
