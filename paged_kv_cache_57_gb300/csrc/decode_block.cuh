// decode_block.cuh -- the per-block step shared by the bf16 decode kernels: one
// 16-token K/V block (TMA-written, 128-byte swizzled boxes of 64 columns) against
// one 16-row tile of rotated queries held as mma.sync A fragments.
//
// S = q' K^T with mma.sync m16n8k16 (bf16 in, fp32 accumulate), then the online
// (max, sum) softmax of "KV Cache, Flash Attention & Otimização de Inferência",
// "Flash Attention -- tiling" (running maximum in log2 units, rescale of the
// running output when it grows), then O += P V with P rounded to bf16.
#pragma once

#include "common.cuh"

namespace lazy {

template <int D>
struct BlockGeom {
  static constexpr int NBOX = D / 64;             // 64-column (128-byte) TMA boxes per row
  static constexpr int BOX_BYTES = kBlock * 128;  // one box: 16 rows x 128 bytes
  static constexpr int KV_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;  // K then V
};

// Issues the TMA loads of one block's K and V rows (kv head kvh) into `stage`,
// completing on `bar`; an id outside the pool is not loaded (the barrier is just
// arrived, and the caller treats the block as empty).
template <int D>
__device__ __forceinline__ void load_block(uint8_t* stage, uint64_t* bar, int phys, int num_pool_blocks, int hkv,
                                           int kvh, const CUtensorMap* kmap, const CUtensorMap* vmap) {
  using G = BlockGeom<D>;
  if (phys < num_pool_blocks) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, G::STAGE_BYTES);
    const int y = (phys * hkv + kvh) * kBlock;
#pragma unroll
    for (int bx = 0; bx < G::NBOX; ++bx) tma_load_2d(stage + bx * G::BOX_BYTES, kmap, bar, bx * 64, y);
#pragma unroll
    for (int bx = 0; bx < G::NBOX; ++bx) tma_load_2d(stage + (G::NBOX + bx) * G::BOX_BYTES, vmap, bar, bx * 64, y);
  } else {
    mbar_arrive(bar);
  }
}

// Issues the TMA loads of one block's e4m3 K and V rows (kv head kvh, d = 128: one
// 16-row x 128-byte box each) into `stage`; an id outside the pool is not loaded.
__device__ __forceinline__ void load_block_fp8(uint8_t* stage, uint64_t* bar, int phys, int num_pool_blocks, int hkv,
                                               int kvh, const CUtensorMap* kmap, const CUtensorMap* vmap) {
  if (phys < num_pool_blocks) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, 2 * kBlock * 128);
    const int y = (phys * hkv + kvh) * kBlock;
    tma_load_2d(stage, kmap, bar, 0, y);
    tma_load_2d(stage + kBlock * 128, vmap, bar, 0, y);
  } else {
    mbar_arrive(bar);
  }
}

// Converts the V box of one landed e4m3 block (K box then V box, 16 rows x 128 bytes,
// 128-byte swizzle: 16-byte chunk c of row r at r * 128 + ((c ^ r) & 7) * 16) into
// an f16 tile at dst laid out as the bf16 path's V tile (per 64-column box of 2048
// bytes, the same swizzle; 4 KB), so that the ldmatrix fragments of
// attend_block_impl read it unchanged (K fragments come from the codes directly).
// Thread tid of nt; a chunk of 16 codes becomes two 16-byte f16 chunks.
__device__ __forceinline__ void convert_fp8_block(const uint8_t* src, uint8_t* dst, int tid, int nt) {
  using G = BlockGeom<128>;
  for (int it = tid; it < kBlock * 8; it += nt) {
    const int r = it >> 3, c = it & 7;
    const uint4 x = *reinterpret_cast<const uint4*>(src + kBlock * 128 + r * 128 + (((c ^ r) & 7) << 4));
    uint4 lo, hi;
    e4m3x4_to_f16x4(x.x, lo.x, lo.y);
    e4m3x4_to_f16x4(x.y, lo.z, lo.w);
    e4m3x4_to_f16x4(x.z, hi.x, hi.y);
    e4m3x4_to_f16x4(x.w, hi.z, hi.w);
    uint8_t* row = dst + (c >> 2) * G::BOX_BYTES + r * 128;
    const int ch = 2 * (c & 3);  // f16 columns 16c .. 16c + 15: chunks ch, ch + 1 of box c / 4
    *reinterpret_cast<uint4*>(row + (((ch ^ r) & 7) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + ((((ch + 1) ^ r) & 7) << 4)) = hi;
  }
}

// Per-lane ldmatrix offsets inside a stage, computed once per kernel. In a box
// written with the 128-byte swizzle, 16-byte chunk c of row r sits at
// (r << 7) | ((c ^ r) & 7) << 4. A lane's chunk for k-step ks is 2 ks plus a
// lane bit, so its offset is the lane constant below XOR ((2 ks) & 7) << 4
// (bits 4-6 only), plus 2048 bytes per 64-column box.
struct LdsmLane {
  uint32_t k;  // K tile (B operand of S = q' K^T), keys (mat >> 1) * 8 + lane % 8
  uint32_t v;  // V tile (transposed B operand of O += P V), keys (mat & 1) * 8 + lane % 8
};

__device__ __forceinline__ LdsmLane ldsm_lane(int lane) {
  const uint32_t mat = (uint32_t)lane >> 3;
  const uint32_t kk = (mat >> 1) * 8 + (lane & 7);
  const uint32_t vk = (mat & 1) * 8 + (lane & 7);
  LdsmLane r;
  r.k = (kk << 7) + ((((mat & 1) ^ kk) & 7) << 4);
  r.v = (vk << 7) + ((((mat >> 1) ^ vk) & 7) << 4);
  return r;
}

// The running maximum is refreshed only when a block's maximum exceeds it by
// more than this (log2 units): weights then stay below 2^8, and the output and
// sum are rescaled rarely.
constexpr float kDecodeRescaleLog2 = 8.f;

// One block for the warp's 16-row tile: rows g = lane/4 and g + 8 hold the
// running state (reference maximum m_r and sum l_r per row, o in accumulator
// layout). The query fragments carry the softmax scale and log2(e), so scores
// come out in log2 units. Only the first `nvalid` slots of the block are keys;
// the others (holes, an unloaded block) get weight 0 and their V rows are masked
// out of the product. With BIAS, row g + 8 rr's score of key k also gets
// bias0[rr] + slope[rr] * k (log2 units; the ALiBi bias). With F16 the operands
// (q fragments, the K/V tiles, P) are f16 instead of bf16 and every score is
// multiplied by sscale first (the FP8-KV decode: the tiles hold unscaled e4m3
// values, sscale is the K scale).
//
// With KFP8 (D = 128, implies F16) kbase is the block's e4m3 K box (16 rows x 128
// bytes, 128-byte swizzle) and the K fragments are converted from it directly; the
// q fragments then follow the permuted head-dimension order of build_q_frags_perm
// (k-step ks, fragment column 2t + {0,1} / 2t + 8 + {0,1} is dimension
// 32t + 4ks + {0,1} / {2,3}), so each lane's four codes of a k-step are one word. V
// comes from the f16 tile at vbase.
template <int D, bool BIAS, bool F16 = false, bool KFP8 = false>
__device__ __forceinline__ void attend_block_impl(uint32_t kbase, LdsmLane ln, const uint32_t (&qa)[D / 16][4],
                                                  int nvalid, float (&o)[D / 8][4], float (&m_r)[2], float (&l_r)[2],
                                                  int lane, const float* bias0, const float* slope,
                                                  float sscale = 1.f, uint32_t vbase = 0) {
  static_assert(!KFP8 || (F16 && D == 128), "e4m3 K fragments: f16 operands, d = 128");
  auto mma = [](float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (F16) mma_16816_f16(d, a, b0, b1);
    else mma_16816(d, a, b0, b1);
  };
  using G = BlockGeom<D>;
  const int t = lane & 3;
  const uint32_t ka = kbase + ln.k;
  const uint32_t va = (KFP8 ? vbase : kbase + G::KV_BYTES) + ln.v;
  // S = q' K^T for the 16 keys: two n-tiles of 8 keys, each summed in two
  // independent chains (even and odd k-steps) to halve the dependent MMA latency.
  float sc[2][2][4];
#pragma unroll
  for (int n = 0; n < 2; ++n)
#pragma unroll
    for (int c = 0; c < 2; ++c) sc[n][c][0] = sc[n][c][1] = sc[n][c][2] = sc[n][c][3] = 0.f;
  if constexpr (KFP8) {
    // keys g and g + 8 (rows of the box; (g + 8) & 7 == g), 16-byte chunks 2t and 2t + 1
    const int g8 = lane >> 2;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t sw = (uint32_t)(((2 * t + h) ^ g8) & 7) << 4;
      const uint4 k0 = lds_v4(kbase + g8 * 128 + sw), k1 = lds_v4(kbase + (g8 + 8) * 128 + sw);
      const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w}, w1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ks = 4 * h + e;
        uint32_t b0, b1, c0, c1;
        e4m3x4_to_f16x4(w0[e], b0, b1);
        e4m3x4_to_f16x4(w1[e], c0, c1);
        mma(sc[0][ks & 1], qa[ks], b0, b1);
        mma(sc[1][ks & 1], qa[ks], c0, c1);
      }
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t r[4];
      ldsm_x4(r, (ka ^ (uint32_t)(((2 * ks) & 7) << 4)) + (ks >> 2) * G::BOX_BYTES);
      mma(sc[0][ks & 1], qa[ks], r[0], r[1]);
      mma(sc[1][ks & 1], qa[ks], r[2], r[3]);
    }
  }
  // sv[rr][e]: row g + 8 rr, key (e >> 1) * 8 + 2t + (e & 1).
  float sv[2][4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int e = 0; e < 4; ++e) sv[rr][e] = sc[e >> 1][0][2 * rr + (e & 1)] + sc[e >> 1][1][2 * rr + (e & 1)];
  if constexpr (F16) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[rr][e] *= sscale;
  }
  if constexpr (BIAS) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[rr][e] += fmaf(slope[rr], (float)((e >> 1) * 8 + 2 * t + (e & 1)), bias0[rr]);
  }
  const bool partial = nvalid < kBlock;  // warp-uniform
  if (partial) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = (e >> 1) * 8 + 2 * t + (e & 1);
      if (key >= nvalid) sv[0][e] = sv[1][e] = -INFINITY;
    }
  }
  uint32_t pa[4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    float mx = fmaxf(fmaxf(sv[rr][0], sv[rr][1]), fmaxf(sv[rr][2], sv[rr][3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (mx > m_r[rr] + kDecodeRescaleLog2) {  // first valid key, or a much larger score
      const float alpha = fast_ex2(m_r[rr] - mx);  // 0 while the row had no key
      m_r[rr] = mx;
      l_r[rr] *= alpha;
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        o[j][2 * rr] *= alpha;
        o[j][2 * rr + 1] *= alpha;
      }
    }
    const float mu = m_r[rr] == -INFINITY ? 0.f : m_r[rr];
    const uint32_t lo = pack_op2<F16>(fast_ex2(sv[rr][0] - mu), fast_ex2(sv[rr][1] - mu));
    const uint32_t hi = pack_op2<F16>(fast_ex2(sv[rr][2] - mu), fast_ex2(sv[rr][3] - mu));
    pa[rr] = lo;      // keys 2t, 2t+1     (a0 / a1)
    pa[2 + rr] = hi;  // keys 8+2t, 8+2t+1 (a2 / a3)
    // The row sum uses the same rounded weights as the product.
    l_r[rr] += sum_op2<F16>(lo) + sum_op2<F16>(hi);
  }
  // O += P V: V^T fragments via ldmatrix.trans, two d-tiles per load.
  if (!partial) {
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r[4];
      ldsm_x4_trans(r, (va ^ (uint32_t)(((2 * c) & 7) << 4)) + (c >> 2) * G::BOX_BYTES);
      mma(o[2 * c], pa, r[0], r[1]);
      mma(o[2 * c + 1], pa, r[2], r[3]);
    }
  } else {  // hole slots may hold anything (even NaN): zero their V
    const int k0 = 2 * t;
    const uint32_t m0 = (k0 < nvalid ? 0x0000ffffu : 0u) | (k0 + 1 < nvalid ? 0xffff0000u : 0u);
    const uint32_t m1 = (k0 + 8 < nvalid ? 0x0000ffffu : 0u) | (k0 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r[4];
      ldsm_x4_trans(r, (va ^ (uint32_t)(((2 * c) & 7) << 4)) + (c >> 2) * G::BOX_BYTES);
      mma(o[2 * c], pa, r[0] & m0, r[1] & m1);
      mma(o[2 * c + 1], pa, r[2] & m0, r[3] & m1);
    }
  }
}

template <int D>
__device__ __forceinline__ void attend_block(uint32_t kbase, LdsmLane ln, const uint32_t (&qa)[D / 16][4], int nvalid,
                                             float (&o)[D / 8][4], float (&m_r)[2], float (&l_r)[2], int lane) {
  attend_block_impl<D, false>(kbase, ln, qa, nvalid, o, m_r, l_r, lane, nullptr, nullptr);
}

template <int D>
__device__ __forceinline__ void attend_block_bias(uint32_t kbase, LdsmLane ln, const uint32_t (&qa)[D / 16][4],
                                                  int nvalid, float (&o)[D / 8][4], float (&m_r)[2], float (&l_r)[2],
                                                  int lane, const float (&bias0)[2], const float (&slope)[2]) {
  attend_block_impl<D, true>(kbase, ln, qa, nvalid, o, m_r, l_r, lane, bias0, slope);
}

// The FP8-KV decode: K fragments from the e4m3 box at kcodes, V from the f16 tile at
// vbase, f16 operands, scores scaled by kscale.
__device__ __forceinline__ void attend_block_fp8(uint32_t kcodes, uint32_t vbase, LdsmLane ln,
                                                 const uint32_t (&qa)[8][4], int nvalid, float (&o)[16][4],
                                                 float (&m_r)[2], float (&l_r)[2], int lane, float kscale) {
  attend_block_impl<128, false, true, true>(kcodes, ln, qa, nvalid, o, m_r, l_r, lane, nullptr, nullptr, kscale,
                                            vbase);
}

// Per-lane description of one logical block: physical id (num_pool_blocks for a
// block that must not be loaded), document start and valid slots.
struct LaneBlock {
  int phys, p, nv;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait: every lane polls, and the warp gives up together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  const bool ok = mbar_wait(bar, parity, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Named barrier of team t (ids 1..4; 0 is __syncthreads) over the team's n threads,
// with an AND of `ok` over them: a warp whose wait gave up makes the whole team
// leave together, so no teammate is left at a barrier the others never reach.
// Literal ids let the compiler see which barriers a kernel uses.
__device__ __forceinline__ bool team_and(int t, int n, bool ok) {
  uint32_t r;
  const uint32_t v = ok ? 1u : 0u;
#define LAZY_TEAM_AND(ID)                                                                                      \
  asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, " #ID                 \
               ", %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"                                                       \
               : "=r"(r)                                                                                       \
               : "r"(v), "r"(n)                                                                                \
               : "memory")
  switch (t) {
    case 0: LAZY_TEAM_AND(1); break;
    case 1: LAZY_TEAM_AND(2); break;
    case 2: LAZY_TEAM_AND(3); break;
    default: LAZY_TEAM_AND(4); break;
  }
#undef LAZY_TEAM_AND
  return r != 0;
}

}  // namespace lazy
