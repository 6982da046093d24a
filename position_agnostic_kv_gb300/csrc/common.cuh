// Shared device and host helpers of liblazykv (sm_103a).
//
// Sources for the method: the LazyAttention pages -- papernotes.org reading note
// ([NOTE] 关键设计, 整体框架, 通用性) and the gist.science summary ([GIST] Implementazione
// Tecnica).  Everything here is written from their statement of the method and from the PTX
// ISA; no code was taken from any implementation.
#pragma once

#include <cstdint>
#include <cstdio>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "lazykv.h"

namespace lazykv {

constexpr int kPage = LAZY_PAGE_SIZE;  // tokens per physical page
constexpr int kMaxHalf = 64;           // rotary_dim / 2 upper bound (D <= 128)

// ------------------------------------------------------------------------------------------
// 64-bit block word ([NOTE] 融合 Triton kernel + bit-packed 元数据: block id, offset and mask
// in one register).  Layout: [4:0] n_valid, [15:5] pg, [39:16] Delta, [63:40] physical page.
// ------------------------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t word_nvalid(uint64_t w) { return uint32_t(w & 31u); }
__host__ __device__ __forceinline__ uint32_t word_pg(uint64_t w) { return uint32_t((w >> 5) & 2047u); }
__host__ __device__ __forceinline__ uint32_t word_delta(uint64_t w) { return uint32_t((w >> 16) & 0xFFFFFFu); }
__host__ __device__ __forceinline__ uint32_t word_page(uint64_t w) { return uint32_t(w >> 40); }

// ------------------------------------------------------------------------------------------
// Positional parameters handed to kernels by value.
//   turns[i] = theta_i / (2 pi) as a 64-bit fixed-point fraction of a turn (value * 2^64).
//   For an integer position p, (p * turns[i]) mod 2^64 is exactly the fractional number of
//   turns of the angle p * theta_i (fixed-point phase accumulation, as in direct digital
//   synthesis), so the angle is reduced without error for any p < 2^32 before sin/cos.
// ------------------------------------------------------------------------------------------
enum PosKind : int { kRope = LAZY_POS_ROPE, kYarn = LAZY_POS_YARN, kAlibi = LAZY_POS_ALIBI, kNone = LAZY_POS_NONE,
                     kRopeX = 16 /* kernel-internal: RoPE with partial rotary_dim or interleaved pairs */ };

struct PosParams {
  int kind;              // PosKind
  int rotary_dim;        // rotated dimensions (a multiple of 16, <= D); the rest pass through
  int interleaved;       // pairs (2i, 2i+1) instead of (i, i + rotary_dim/2)
  float scale_log2;      // softmax scale * log2(e): logits are kept in base-2 units
  const float* slopes;   // ALiBi slopes [Hq] (device) or null
  const float* table;    // cos/sin table [max_pos][rotary_dim] (device) or null
  int max_pos;
  unsigned long long turns[kMaxHalf];
};

// sin and cos of the angle p * theta, with theta given as fixed-point turns.
__device__ __forceinline__ void turn_sincos(uint32_t p, unsigned long long turns, float& s, float& c) {
  const unsigned long long frac = (unsigned long long)p * turns;  // mod 2^64 = fractional turns
  const int hi = int(uint32_t(frac >> 32));                        // [-2^31, 2^31): [-1/2, 1/2) turn
  const float half_turns = float(hi) * 4.656612873077393e-10f;     // * 2^-31 -> [-1, 1)
  sincospif(half_turns, &s, &c);                                     // sin/cos(pi * x)
}

// The same angle through the SFU's sine and cosine (__sincosf).  The exact turn count leaves
// an argument in [-pi, pi), where the hardware approximation is good to about 1e-6 absolute,
// far below the rounding the rotated value gets next in the attention kernels (an f16 operand
// of the tensor cores, or an fp32 query); the stored keys (kv_write) and the cos/sin table keep
// the correctly rounded sincospif.
__device__ __forceinline__ void turn_sincos_fast(uint32_t p, unsigned long long turns, float& s, float& c) {
  const unsigned long long frac = (unsigned long long)p * turns;
  const int hi = int(uint32_t(frac >> 32));
  __sincosf(float(hi) * 1.4629180792671596e-9f, &s, &c);  // * pi * 2^-31 -> [-pi, pi)
}

// 2^x on the SFU (ex2.approx, flush-to-zero; 2^-inf = 0), for softmax weights.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------------------------------
// bf16 <-> fp32
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
__device__ __forceinline__ float2 bf2_to_f2(uint32_t x) { return make_float2(bf_lo(x), bf_hi(x)); }
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------------------------------------
// Shared memory, mbarrier and bulk-copy wrappers (PTX ISA: mbarrier, cp.async.bulk).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return uint32_t(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait is bounded: after ~kWaitNs without progress the caller gets false, records
// LAZY_STATUS_TIMEOUT and leaves; the kernel never spins forever.
constexpr uint64_t kWaitNs = 1500000000ull;  // 1.5 s

// Time spent in one wait, from successive readings of the global timer.  Each reading adds
// the step since the previous one clamped to [20 ns, 1 ms], so a jump of the timer (forwards
// or backwards) cannot end a wait early, and a timer that stood still would still end it.
struct WaitClock {
  uint64_t last, spent;
  __device__ __forceinline__ WaitClock() : last(global_ns()), spent(0) {}
  __device__ __forceinline__ bool expired() {
    const uint64_t now = global_ns();
    const uint64_t d = now - last;  // a backwards jump wraps to a huge step, clamped below
    last = now;
    spent += d < 20ull ? 20ull : (d > 1000000ull ? 1000000ull : d);
    return spent > kWaitNs;
  }
};

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  WaitClock clk;
  while (true) {
    if (mbar_test(bar, parity)) return true;
    if (clk.expired()) return false;
  }
}

// Bulk (non-tensor) asynchronous copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Programmatic dependent launch (PTX griddepcontrol).  Every kernel of the library is launched
// so that it may become resident while the previous kernel of the stream drains; it calls
// pdl_wait() before it reads or writes any global memory (that returns once the previous grid
// has completed and its writes are visible), and pdl_trigger() once every one of its CTAs is
// running, which lets the next kernel of the stream start its launch early.  Both are no-ops
// when the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint64_t ldg_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// ------------------------------------------------------------------------------------------
// Host side
// ------------------------------------------------------------------------------------------
int fail(int code, const char* fmt, ...);  // records a thread-local message, returns code
int check_device();                        // LAZY_EARCH unless CC 10.x
int sm_count();                            // current device
uint32_t* status_word();                   // device address of the status word (current device)
int prepare_pos(const lazy_pos_cfg* cfg, int Hq, int D, float scale, PosParams* out);

// Launch `kern` on `st` with programmatic stream serialisation (see pdl_wait above).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

#define LAZY_CUDA_TRY(expr)                                                              \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess)                                                               \
      return ::lazykv::fail(LAZY_ECUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

}  // namespace lazykv
