// common.cuh -- device helpers shared by the LazyAttention kernels (sm_103a).
//
// Everything here is plain inline PTX or CUDA intrinsics: mbarrier pipelines with
// bounded waits, TMA tile loads, ldmatrix / mma.sync fragments, the packed block
// word, and the rotation table lookup.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lazy_attn.h"

namespace lazy {

constexpr int kBlock = 16;             // tokens per physical block
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: any pipeline wait longer than this is a fault

// ------------------------------------------------------------------ status word

__device__ __forceinline__ void raise_status(unsigned int* status, unsigned int bit) {
  if (status) atomicOr(status, bit);
}

// ------------------------------------------------------------------ addresses / timers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA / tensor core).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same condition (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after
// limit_ns (kWaitLimitNs unless a test asks for less), sets LAZY_DEV_TIMEOUT and
// returns false: callers then skip the rest of their work, so the kernel always
// terminates.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      raise_status(status, LAZY_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on `bar`
// as transaction bytes. x is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a box written by TMA
// with CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, box base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return (r << 7) | (((c ^ r) & 7u) << 4); }

// ------------------------------------------------------------------ warp-level MMA

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same product with f16 inputs (the FP8-KV decode: e4m3 values are exact in f16).
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four e4m3 bytes (byte i = element i) to two f16x2 words (elements 0,1 and 2,3,
// element 0 in the low half). Every e4m3 value, subnormals and zeros included, is
// exact in f16, so the conversion is exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 2^x on the SFU (PTX ex2.approx, flush-to-zero); 2^-inf = +0.
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packs two operands of the 16-bit MMA type: f16 when F16, else bf16.
template <bool F16>
__device__ __forceinline__ uint32_t pack_op2(float lo, float hi) {
  if constexpr (F16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

// The two values of a packed operand word, as fp32.
template <bool F16>
__device__ __forceinline__ float sum_op2(uint32_t w) {
  if constexpr (F16) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    return f.x + f.y;
  } else {
    return __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
  }
}

// ------------------------------------------------------------------ block words

struct BlockInfo {
  int phys;    // physical block id
  int p;       // global start position of the block's document
};

__device__ __forceinline__ BlockInfo decode_word(uint32_t w, int b, int id_bits) {
  BlockInfo bi;
  bi.phys = static_cast<int>(w & ((1u << id_bits) - 1u));
  const int off = static_cast<int>(w) >> id_bits;  // arithmetic shift: signed field
  bi.p = kBlock * b - off;
  return bi;
}

// Valid slots of logical block b (see the layout notes in lazy_attn.h).
__device__ __forceinline__ int block_valid(int b, int nb, int seq_len, int p_b, int p_next) {
  if (b == nb - 1) return seq_len - kBlock * (nb - 1);
  if (p_next != p_b) return ((p_next - p_b - 1) & (kBlock - 1)) + 1;
  return kBlock;
}

// ------------------------------------------------------------------ rotation

// (cos, sin)(delta * w) for a frequency given in turns, t = w / (2 pi), stored as
// t.x + t.y. The product delta * t.x is split exactly into ph + pe (error-free
// product with one FMA); ph - rint(ph) is exact in fp32, so the fraction of a
// turn is formed with two small roundings and sincospif evaluates it without a
// range reduction. |angle error| is below about 5e-7 rad for |delta| < 2^24.
__device__ __forceinline__ float2 rope_cs(float2 t, int delta, unsigned int* status) {
  if (delta >= LAZY_MAX_ROPE_OFFSET || delta <= -LAZY_MAX_ROPE_OFFSET) {
    raise_status(status, LAZY_DEV_POS_RANGE);
    delta = delta > 0 ? LAZY_MAX_ROPE_OFFSET - 1 : -(LAZY_MAX_ROPE_OFFSET - 1);
  }
  const float n = static_cast<float>(delta);  // exact: |delta| < 2^24
  const float ph = n * t.x;
  const float pe = fmaf(n, t.x, -ph);  // n * t.x == ph + pe exactly
  const float f = (ph - rintf(ph)) + (pe + n * t.y);
  float s, c;
  sincospif(2.f * f, &s, &c);
  return make_float2(c, s);
}

}  // namespace lazy
