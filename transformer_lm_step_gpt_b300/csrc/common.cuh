// common.cuh -- device helpers shared by the kernels of libgpt2.so.
//
// Types, warp reductions, the device error word, and thin inline-PTX
// wrappers (mbarrier, TMA bulk tensor copies, tcgen05) written from the
// public PTX ISA.  Every wait on an mbarrier is bounded by the global
// SM cycle counter: on expiry the waiting thread records a timeout in the
// error word and returns false, and the kernel winds down without trapping.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

typedef __nv_bfloat16 bf16;

// Bits of the device error word (one int per model, read back by the host
// at synchronising calls).
enum : int {
  DEVERR_TOKEN = 1,    // a token / target id outside [0, V)
  DEVERR_TIMEOUT = 2,  // a bounded wait expired
};

// A bounded wait gives up after this many SM clock cycles: 2 s at the
// B300's top SM clock (2,032 MHz), under 4 s at 1 GHz.  The SM's own cycle
// counter is read (a few cycles) rather than the global nanosecond timer,
// whose reads are slow enough to delay every wait that is not already
// complete on its first test.
#define GPT2_WAIT_LIMIT_CYCLES 4000000000ll

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ long long sm_cycles() { return clock64(); }

__device__ __forceinline__ void record_error(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// GELU, tanh form: x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), and its
// derivative; tanhf is CUDA's own.
#define GELU_S 0.7978845608028654f
#define GELU_A 0.044715f
__device__ __forceinline__ float gelu_f(float x) {
  return 0.5f * x * (1.f + tanhf(GELU_S * (x + GELU_A * x * x * x)));
}
__device__ __forceinline__ float gelu_grad_f(float x) {
  const float th = tanhf(GELU_S * (x + GELU_A * x * x * x));
  return 0.5f * (1.f + th) + 0.5f * x * (1.f - th * th) * GELU_S * (1.f + 3.f * GELU_A * x * x);
}

// The same two functions with the hardware tanh approximation (PTX
// tanh.approx.f32, relative error about 2^-11), for results that are
// rounded to bf16 anyway.
__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float gelu_hw(float x) {
  return 0.5f * x * (1.f + tanh_hw(GELU_S * (x + GELU_A * x * x * x)));
}
// gelu(x) and gelu'(x) from one tanh.approx, the products regrouped so that
// nine FP32 operations remain: with x2 = x^2, u = x (S + S A x2),
// th = tanh u, h = (1 + th) / 2:
//   gelu(x)  = x h
//   gelu'(x) = h + x (1 - th^2) (S/2 + 3 S A x2 / 2)
__device__ __forceinline__ void gelu_and_grad_hw(float x, float& g, float& gd) {
  const float x2 = x * x;
  const float th = tanh_hw(x * fmaf(GELU_S * GELU_A, x2, GELU_S));
  const float h = fmaf(0.5f, th, 0.5f);
  g = x * h;
  const float w = fmaf(1.5f * GELU_S * GELU_A, x2, 0.5f * GELU_S);
  gd = fmaf(x * w, fmaf(-th, th, 1.f), h);
}

// 2^x with the PTX ex2.approx.ftz.f32 instruction (relative error about
// 2^-22; inputs below -126 flush to 0), for probabilities that are rounded
// to bf16 or summed in fp32.
__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pairs of fp32 values in one 64-bit register and the PTX .f32x2
// arithmetic (sm_100 and later): one instruction for two elements, which
// halves the issue slots that elementwise warps take from the single
// thread that issues a kernel's tensor-core instructions.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (PTX three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Named barrier `id` (1..15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation (launch_pdl in kernels.h): it lets
// the next kernel in the stream start launching (pdl_trigger) and, before it
// touches any global memory, waits until the previous kernel has completed
// and its writes are visible (pdl_wait).  Both are no-ops for a kernel
// launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same test, but a thread whose phase has not completed is suspended
// until it completes or about `ns` nanoseconds pass.  A waiting thread then
// issues nothing: a polling loop without the hint takes issue slots from
// the warps that share its scheduler (measured: it halved the rate of the
// attention kernels' elementwise warps and MMA issue).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records a timeout) if the time limit passes first.  Between
// tests only the SM cycle counter is read: the error word (global memory)
// is looked at about once per 2^20 cycles, so that a wait whose phase
// completes is not held up behind a load from L2.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = sm_cycles();
  long long check = t0 + (1ll << 20);
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 1000000u)) return true;
    const long long t = sm_cycles();
    if (t > check) {
      // once any wait of the launch has given up, the others stop early
      // instead of each spending the full limit
      if (err && (*reinterpret_cast<volatile int*>(err) & DEVERR_TIMEOUT)) return false;
      if (t - t0 > GPT2_WAIT_LIMIT_CYCLES) {
        record_error(err, DEVERR_TIMEOUT);
        return false;
      }
      check = t + (1ll << 20);
    }
  }
}

// ------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// ------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M rows = TMEM lanes, K bf16 packed
// two per 32-bit column, K-step kk at column a_tmem + 8 kk) comes from tensor
// memory instead of shared memory.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four consecutive K steps in one statement (one predicate set-up for all
// four): D (+)= A_k B_k^T for k = 0..3 with shared-memory descriptors
// a + k*AS and b + k*BS (AS, BS: the K step's byte offset / 16); the first
// accumulates iff acc != 0, the others always.  The issuing thread then
// spends about one instruction per MMA, which matters when it shares its
// scheduler with busy elementwise warps.
template <int AS, int BS>
__device__ __forceinline__ void tc_mma4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a1, a2, a3, b1, b2, b3;\n"
      " setp.ne.b32 p, %3, 0;\n setp.eq.b32 t, %3, %3;\n"
      " add.s64 a1, %1, %5;\n add.s64 a2, %1, %6;\n add.s64 a3, %1, %7;\n"
      " add.s64 b1, %2, %8;\n add.s64 b2, %2, %9;\n add.s64 b3, %2, %10;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %4, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %4, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %4, t;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(acc), "r"(idesc), "n"(AS), "n"(2 * AS), "n"(3 * AS), "n"(BS), "n"(2 * BS), "n"(3 * BS)
      : "memory");
}
// The same with A in tensor memory: columns a, a+8, a+16, a+24 (K = 16
// bf16 values packed in 8 columns per step).
template <int BS>
__device__ __forceinline__ void tc_mma4_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 b1, b2, b3;\n"
      " setp.ne.b32 p, %3, 0;\n setp.eq.b32 t, %3, %3;\n"
      " add.s64 b1, %2, %5;\n add.s64 b2, %2, %6;\n add.s64 b3, %2, %7;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+8], b1, %4, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+16], b2, %4, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+24], b3, %4, t;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(acc), "r"(idesc), "n"(BS), "n"(2 * BS), "n"(3 * BS)
      : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 columns of 32-bit words: thread i of the warp receives lane
// (base lane + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// The same for 16, 8 and 4 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
// N consecutive columns (N = 4, 8, 16, 32 or a multiple of 32) into r[0..N).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 4) tmem_ld4(taddr, r);
  else if constexpr (N == 8) tmem_ld8(taddr, r);
  else if constexpr (N == 16) tmem_ld16(taddr, r);
  else {
    static_assert(N % 32 == 0, "column count");
#pragma unroll
    for (int i = 0; i < N / 32; i++) tmem_ld32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
  }
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// thread i of the warp writes 16 32-bit words to lane (base lane + i),
// columns col .. col+15
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
// N consecutive columns (N = 4, 8 or a multiple of 16) from r[0..N).
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  if constexpr (N == 4) tmem_st4(taddr, r);
  else if constexpr (N == 8) tmem_st8(taddr, r);
  else {
    static_assert(N % 16 == 0, "column count");
#pragma unroll
    for (int i = 0; i < N / 16; i++) tmem_st16(taddr + 16 * i, r + 16 * i);
  }
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Make generic-proxy shared-memory writes (plain st.shared) visible to the
// async proxy (tcgen05.mma operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMA store / reduce-add of a shared-memory box into a 2-D or 3-D tensor
// (bulk-group completion), and the waits on outstanding groups.
// Contiguous bulk copy global -> shared (both 16-byte aligned, bytes a
// multiple of 16), completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(tmap),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, const void* src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tmap),
      "r"(smem_u32(src)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the shared-memory sources of all committed groups have been read
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until all committed groups have completed
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// tcgen05 shared-memory matrix descriptor for a 128-byte-swizzled operand
// whose swizzle atoms (8 rows x 128 B) start on 1024-byte boundaries.
//   K-major operand:  8-row groups SBO bytes apart; LBO unused (16).
//   MN-major operand: 64-element MN blocks LBO bytes apart, 8-row K groups
//                     SBO bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16,
// shape M x N (M = 64 or 128 for one CTA), each operand K- or MN-major.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// kind::f8f6f4 with E4M3 A and B (format code 0 in the A / B fields), fp32
// accumulator, both operands K-major.
__host__ __device__ constexpr uint32_t tc_idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------ cross-CTA flags
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// order this thread's generic-proxy accesses against its async-proxy (TMA)
// accesses of global memory
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Bounded wait until *p == want (another CTA's release); records a timeout
// and gives up like mbar_wait.
__device__ __forceinline__ bool flag_wait(const int* p, int want, int* err) {
  if (ld_acquire_gpu(p) == want) return true;
  const long long t0 = sm_cycles();
  for (uint32_t i = 0;; i++) {
    __nanosleep(64);  // leave the issue slots to the warps that share the scheduler
    if (ld_acquire_gpu(p) == want) return true;
    if ((i & 63u) == 63u) {
      if (err && (*reinterpret_cast<volatile int*>(err) & DEVERR_TIMEOUT)) return false;
      if (sm_cycles() - t0 > GPT2_WAIT_LIMIT_CYCLES) {
        record_error(err, DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------ CTA pairs
// A cluster of two CTAs on the two SMs of a TPC drives one M=256 MMA
// (tcgen05 cta_group::2): each CTA holds half of A (its 128 rows), half of
// B (N/2 rows) and its 128 accumulator lanes; one thread of the even CTA
// (the leader) issues the MMAs.  Every tcgen05 instruction of such a kernel
// that takes a cta_group uses cta_group::2.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs; release/acquire orders shared-memory writes
// (mbarrier initialisation included) across the pair.  Not .aligned, so a
// warp may arrive diverged.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr) : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA (cl_bar: cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* tmap, uint32_t cl_bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(cl_bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with E4M3 operands (kind::f8f6f4, one byte per element; a K
// step of one instruction is 32 elements = 32 bytes, as for kind::f16).
__device__ __forceinline__ void tc_mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at this shared-memory offset in both CTAs of the
// pair once all previously issued pair MMAs of this thread have completed.
__device__ __forceinline__ void tc_commit_pair_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
