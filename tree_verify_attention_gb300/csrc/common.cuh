// Shared device helpers of libdfv (sm_103a): status reporting, bounded
// mbarrier waits, 1-D bulk copies (TMA engine), ldmatrix and mma.sync
// wrappers. Inline PTX is hand-written here.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dfv.h"

namespace dfv {

constexpr int kMaxNodes = DFV_MAX_NODES;
constexpr int kMaskWords = (kMaxNodes + 31) / 32;   // 3
// Every wait in the library gives up after kWaitNs nanoseconds of the GPU's
// global timer (far above any step's duration) and sets DFV_DEV_TIMEOUT;
// kWaitPolls bounds the polls as well, in case the timer stood still.
constexpr uint64_t kWaitNs = 100ull * 1000 * 1000;   // 100 ms
constexpr uint32_t kWaitPolls = 1u << 30;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Polls `done()` until it returns true (then true) or the time limit
// passes (then false). The timer is read once every 64 polls.
template <typename F>
__device__ __forceinline__ bool wait_bounded(F done) {
  if (done()) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < kWaitPolls; it += 64) {
#pragma unroll 1
    for (int k = 0; k < 64; ++k)
      if (done()) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

// Named CTA barrier `id` (1..15) over `count` threads (a multiple of 32):
// sync waits for all of them, arrive counts this thread without waiting.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// sync on named barrier `id` that also returns whether `v` held in every
// one of the `count` threads.
__device__ __forceinline__ bool named_sync_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void report(uint32_t* status, uint32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch (PTX griddepcontrol). launch_dependents:
// the next kernel of the stream, if it was launched with programmatic stream
// serialisation, may start its CTAs once every CTA of this grid has issued
// it or exited. wait: blocks until the grids this one depends on have
// completed and their memory operations are visible. Both are no-ops for a
// plain launch.
__device__ __forceinline__ void grid_dep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One poll of phase `parity`; true once that phase has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (kWaitNs); false if the limit was reached.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  return wait_bounded([&]() { return mbar_try_wait(bar, parity); });
}

// 1-D bulk copy global -> shared through the TMA engine, completing
// `bytes` of transaction count on `bar`. dst, src 16-byte aligned; bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy shared -> global through the TMA engine, in this thread's
// bulk async-group; bulk_commit_wait() commits the group and waits until its
// writes are complete. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_wait() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Orders this thread's global accesses through the generic proxy with those
// through the async proxy (bulk copies), both ways.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- tensor core (legacy path)

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

// D += A * B, m16n8k16, f16 inputs, f32 accumulators.
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- Q4_0

// Dequantise the 16 code bytes + fp16 scale of one Q4_0 block into 32 fp16
// values (q - 8) * d: the integer (q - 8) is exact in fp16, the product is
// rounded once to nearest. `codes` is 2-byte aligned.
__device__ __forceinline__ void q4_0_block_to_half(const uint16_t* codes, __half d,
                                                   __half* out_lo16, __half* out_hi16) {
  const __half2 d2 = __halves2half2(d, d);
  const __half2 bias = __float2half2_rn(1032.0f);  // 1024 + 8
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t u = codes[k];                   // bytes 2k (low), 2k+1 (high)
    // 0x6400 | n is the fp16 value 1024 + n for n in [0, 15]
    const uint32_t lo = 0x64006400u | (u & 0x000Fu) | ((u & 0x0F00u) << 8);
    const uint32_t hi = 0x64006400u | ((u >> 4) & 0x000Fu) | ((u & 0xF000u) << 4);
    __half2 vlo = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo), bias), d2);
    __half2 vhi = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&hi), bias), d2);
    *reinterpret_cast<__half2*>(out_lo16 + 2 * k) = vlo;
    *reinterpret_cast<__half2*>(out_hi16 + 2 * k) = vhi;
  }
}

// Quantise 32 float values to one Q4_0 block with the binary32 rule:
// m = first element of largest magnitude, d = m / -8, id = 1/d (0 if d = 0),
// code = min(15, trunc(RN(RN(x * id) + 8.5))); scale stored as fp16 RN(d).
// Results in registers: the 16 code bytes as four little-endian words (byte
// j = code j | code j+16 << 4) and the fp16 scale bits.
__device__ __forceinline__ void q4_0_quantize_regs(const float* x, uint32_t* code, uint32_t& dbits) {
  float amax = -1.0f, m = 0.0f;
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float a = fabsf(x[k]);
    if (a > amax) { amax = a; m = x[k]; }
  }
  const float d = __fdiv_rn(m, -8.0f);
  const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
  uint32_t q[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float t = __fadd_rn(__fmul_rn(x[k], id), 8.5f);
    const int c = __float2int_rz(t);
    q[k] = static_cast<uint32_t>(c < 15 ? c : 15);
  }
  dbits = __half_as_ushort(__float2half_rn(d));
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = 4 * w + b;
      word |= (q[j] | (q[j + 16] << 4)) << (8 * b);
    }
    code[w] = word;
  }
}

// The same block written as 18 bytes (fp16 scale, then the 16 code bytes).
__device__ __forceinline__ void q4_0_quantize_block(const float* x, uint8_t* blk) {
  uint32_t code[4], dbits;
  q4_0_quantize_regs(x, code, dbits);
  uint16_t* w = reinterpret_cast<uint16_t*>(blk);   // blocks are 2-byte aligned
  w[0] = static_cast<uint16_t>(dbits);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w[1 + 2 * k] = static_cast<uint16_t>(code[k] & 0xFFFFu);
    w[2 + 2 * k] = static_cast<uint16_t>(code[k] >> 16);
  }
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for
// this thread's copies (they then are visible to the thread).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Eight bf16 values (16 bytes) as eight binary16 values, each rounded to
// nearest even (exact for bf16 values in the binary16 normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8_rn(uint4 v) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint4 o;
  uint32_t* ov = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(b[e]);
    const __half2 h = __floats2half2_rn(f.x, f.y);
    ov[e] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return o;
}

// Bytes of one cache row (one KV head, one position) of D values.
__host__ __device__ constexpr int kv_row_bytes(int fmt, int D) {
  return fmt == DFV_KV_F16 ? D * 2 : D / 32 * 18;
}

// ---------------------------------------------------------------- host helpers

int sm_count();   // SMs of the current device (cached per device)

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace dfv
