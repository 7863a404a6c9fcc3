// prefill_common.cuh -- pieces shared by the two prefill kernels (one and two
// query tiles per CTA): tile geometry, per-block metadata, the packed-fp32 RoPE
// rotation of 16-byte bf16 chunks, and small wait / exp helpers.
#pragma once

#include "kernels.h"
#include "tcgen05.cuh"

namespace lazy {
namespace pf {

constexpr int BM = 128;                 // query rows per tile (MMA M)
constexpr int BN = 128;                 // keys per tile (MMA N of S)
constexpr int D = 128;                  // head dim
constexpr int BLOCKS = BN / kBlock;     // 8 blocks per key tile
constexpr int HALF = BM * 128;          // one 64-column half of a 128-row tile (bytes)
constexpr int TILE = 2 * HALF;          // 32 KiB
constexpr float RESCALE_LOG2 = 8.f;     // refresh the running max when it grows by more than this

struct KMeta {
  int p;       // document start position
  int nvalid;  // valid slots (0 for blocks past the sequence or with a bad id)
};
struct VMeta {
  int nvalid;
  int chunk_j0;  // chunk-local index of the block's first key, or -1 for cached documents
  int pos;       // the position the block word gives (ALiBi: that of the block's first key)
  int pad;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

// Named barrier `id` (1..15; 0 is __syncthreads) over n threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// The same barrier with an AND reduction of v over the participating threads.
__device__ __forceinline__ bool named_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// 2^x on the SFU (PTX ex2.approx, flush-to-zero); 2^-inf = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Rotation coefficients of 8 consecutive frequencies as packed fp32 pairs
// (cos, sin, -sin), each multiplied by `scale`.
struct Rot8 {
  uint64_t c[4], s[4], ns[4];
};

__device__ __forceinline__ Rot8 make_rot8(const float2 (&cs)[8], float scale) {
  Rot8 r;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 a = cs[2 * k], b = cs[2 * k + 1];
    r.c[k] = f2(a.x * scale, b.x * scale);
    r.s[k] = f2(a.y * scale, b.y * scale);
    r.ns[k] = f2(-a.y * scale, -b.y * scale);
  }
  return r;
}

// Rotates 8 rotate-half pairs held as two 16-byte bf16 chunks (x: dims i, y: dims
// i + 64): x' = x c - y s, y' = y c + x s on packed fp32 pairs, rounded to bf16.
__device__ __forceinline__ void rotate_chunk(uint4& X, uint4& Y, const Rot8& R) {
  uint32_t* xw = reinterpret_cast<uint32_t*>(&X);
  uint32_t* yw = reinterpret_cast<uint32_t*>(&Y);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t x2 = f2(__uint_as_float(xw[k] << 16), __uint_as_float(xw[k] & 0xffff0000u));
    const uint64_t y2 = f2(__uint_as_float(yw[k] << 16), __uint_as_float(yw[k] & 0xffff0000u));
    const float2 xn = f2_split(f2_fma(y2, R.ns[k], f2_mul(x2, R.c[k])));
    const float2 yn = f2_split(f2_fma(x2, R.s[k], f2_mul(y2, R.c[k])));
    xw[k] = pack_bf16x2(xn.x, xn.y);
    yw[k] = pack_bf16x2(yn.x, yn.y);
  }
}

// Query rows of a tile sit at positions base + i, i = 16 k + r < 128. The tile's
// base angles (cos, sin)(base w_f) take one sincospif per frequency per CTA; the
// table rows i = 16 k (k < 8) and i = r (r < 16), 24 rows, are copied to shared
// memory once per CTA; row i's angles then follow by two angle additions (a few
// fp32 operations, about 3 ulp), with no global-memory latency per row.
constexpr int kAngleRows = 24;

__device__ __forceinline__ float2 add_angles(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.y, b.x, a.x * b.y));
}

// Copies the table's rows for offsets 0, 16, ..., 112 (slots 0..7) and 0 .. 15
// (slots 8..23) to sm_rows, frequency-major: entry (f, slot) at f * 24 + slot, so
// that 32 threads rotating 32 consecutive rows read 16 consecutive entries (no bank
// conflict) for the row offset and one broadcast entry for the multiple of 16.
// Thread tid of n.
__device__ __forceinline__ void load_angle_rows(float2* sm_rows, const float2* __restrict__ rope, int tid, int n) {
  const float2* src = rope + D / 2;  // row part of the table: [row][D/2]
  for (int idx = tid; idx < kAngleRows * (D / 2); idx += n) {
    const int f = idx / kAngleRows, slot = idx % kAngleRows;
    const int src_row = slot < 8 ? 16 * slot : slot - 8;
    sm_rows[idx] = __ldg(&src[src_row * (D / 2) + f]);
  }
}

// Rotation coefficients of the 8 frequencies of chunk c for row offset i.
__device__ __forceinline__ Rot8 row_rot8(const float2* base_cs, const float2* sm_rows, int i, int c, float scale) {
  const int s16 = i >> 4, s1 = 8 + (i & 15);
  float2 cs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int f = 8 * c + e;
    cs[e] = add_angles(add_angles(base_cs[f], sm_rows[f * kAngleRows + s16]), sm_rows[f * kAngleRows + s1]);
  }
  return make_rot8(cs, scale);
}

// Rotates chunks [c0, c1) of row i of a 128-row Q tile in place (both 64-column
// halves, 128-byte swizzled) by R_{base+i}, pre-scaled by `scale`.
__device__ __forceinline__ void rotate_q_row(uint8_t* sQ, int i, int c0, int c1, const float2* base_cs,
                                             const float2* sm_rows, float scale) {
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint4 X = *reinterpret_cast<uint4*>(sQ + sw128(i, c));
    uint4 Y = *reinterpret_cast<uint4*>(sQ + HALF + sw128(i, c));
    rotate_chunk(X, Y, row_rot8(base_cs, sm_rows, i, c, scale));
    *reinterpret_cast<uint4*>(sQ + sw128(i, c)) = X;
    *reinterpret_cast<uint4*>(sQ + HALF + sw128(i, c)) = Y;
  }
}

}  // namespace pf
}  // namespace lazy
