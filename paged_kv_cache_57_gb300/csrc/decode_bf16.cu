// decode_bf16.cu -- LazyAttention decode, bf16 pools, split-K over the paged context.
//
// Technical summary "Resumo Técnico: LazyAttention", "Implementação Técnica",
// item 2 (Decoding): the query tile is one row per sequence; the rotation is
// fused into the inner loop and the query is re-rotated only when the relative
// offset changes (a new document); block id and offset travel in one packed
// word; only K and V are read from memory.
//
// One CTA handles one (sequence, KV head, split) and all g = Hq/Hkv query heads
// of that KV head, which become the rows of 16-row mma.sync tiles (the GQA group
// is what turns a 16-token block into a small dense contraction).
//
// The CTA is TEAMS independent teams of MT warps (MT = row tiles of 16 heads).
// Team t owns a contiguous quarter of the split's logical blocks and a ring
// of SPT shared-memory stages; it is its own loader: as soon as it has consumed
// a stage it refills it (one TMA box per 64 columns of K and of V, 128-byte
// swizzle) with its block SPT positions ahead. There is no producer warp and no
// cross-warp hand-off on the load path, so every team keeps SPT blocks in flight.
// Block words are fetched 32 at a time (one per lane), a chunk ahead.
//
// Per block a warp: (re)builds the A fragments of R_{m-p} q when the document
// start p changed (cos/sin evaluated in registers, no memory access), computes
// S = q' K^T and O += P V with mma.sync (bf16 in, fp32 accumulate) and runs the
// online (max, sum) softmax of "KV Cache, Flash Attention & Otimização de
// Inferência", "Flash Attention -- tiling". Teams merge in shared memory with the
// same rescale; a split writes fp32 partials (or, with one split, the final
// output) and decode_combine merges the splits.
#include <cfloat>
#include <climits>
#include <type_traits>

#include "decode_block.cuh"
#include "kernels.h"

#ifndef LAZY_DECODE_SPT
#define LAZY_DECODE_SPT 2  // stages per team (2 lets three 4-warp CTAs share an SM)
#endif

namespace lazy {

// FP8: each ring stage holds one block's e4m3 K and V (one 16-row x 128-byte box each),
// and every team has one more buffer where the block is converted to f16 in the
// bf16 path's tile layout.
template <int D, int MT, int SPT, bool FP8 = false>
struct DecodeCfg {
  static constexpr int TEAMS = (MT >= 4) ? 2 : 4;
  static constexpr int CW = TEAMS * MT;  // warps
  static constexpr int NTHREADS = 32 * CW;
  static constexpr int HALF = D / 2;
  static constexpr int NBOX = D / 64;  // 64-column (128-byte) TMA boxes per row
  static constexpr int BOX_BYTES = kBlock * 128;
  static constexpr int KV_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = FP8 ? 2 * kBlock * D : 2 * KV_BYTES;
  static constexpr int CONV_BYTES = FP8 ? KV_BYTES : 0;  // the f16 V tile
  static constexpr int TEAM_BYTES = SPT * STAGE_BYTES + CONV_BYTES;
  static constexpr int ROWS = MT * 16;
  static constexpr int QS_STRIDE = D + 8;  // fp32 q rows, padded against bank conflicts
  static constexpr int MERGE_BYTES = TEAMS * ROWS * (D + 2) * 4;
  static constexpr int RING_BYTES = TEAMS * TEAM_BYTES;
  static constexpr int STAGES_BYTES =
      ((RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES) + 1023) / 1024 * 1024;
  static constexpr int QS_BYTES = ROWS * QS_STRIDE * 4;
  static constexpr int BAR_BYTES = TEAMS * SPT * 8;
  static constexpr int SMEM = 1024 + STAGES_BYTES + QS_BYTES + BAR_BYTES;
};

__device__ __forceinline__ LaneBlock describe_block(bool live, int b, int nb, int seq_len, uint32_t w, uint32_t wn,
                                                    int id_bits, int num_pool_blocks, unsigned int* status) {
  LaneBlock r{num_pool_blocks, 0, 0};
  if (!live) return r;
  const BlockInfo bi = decode_word(w, b, id_bits);
  const int pn = (b + 1 < nb) ? decode_word(wn, b + 1, id_bits).p : bi.p;
  int nv = block_valid(b, nb, seq_len, bi.p, pn);
  nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
  if (bi.phys >= num_pool_blocks) {
    raise_status(status, LAZY_DEV_BAD_BLOCK_ID);
    nv = 0;
  }
  r.phys = bi.phys < num_pool_blocks ? bi.phys : num_pool_blocks;
  r.p = bi.p;
  r.nv = nv;
  return r;
}

// A fragments of scale * R_delta q for rows (mt*16 + g, mt*16 + g + 8), g = lane/4.
// The thread owns columns 16ks + 2t + {0,1,8,9}; ks and ks + D/32 hold the two
// halves of the same rotate-half pairs, so each pair is rotated by one thread.
// cs_of(ks, i) returns (cos, sin) for frequency i and is called by all lanes
// with the same ks sequence (it may shuffle).
template <int D, int QS_STRIDE, bool F16 = false, typename CsFn>
__device__ __forceinline__ void build_q_frags(uint32_t (&qa)[D / 16][4], const float* __restrict__ qs, int mt,
                                              int lane, float scale, CsFn cs_of) {
  constexpr int HALF = D / 2;
  const int g = lane >> 2, t = lane & 3;
  const float* r0 = qs + (mt * 16 + g) * QS_STRIDE;
  const float* r1 = r0 + 8 * QS_STRIDE;
#pragma unroll
  for (int ks = 0; ks < D / 32; ++ks) {
    float xr[2][4], yr[2][4];
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const int i = 16 * ks + 2 * t + 8 * e2;  // columns i, i+1
      float2 c0 = cs_of(ks, i);
      float2 c1 = cs_of(ks, i + 1);
      c0.x *= scale, c0.y *= scale, c1.x *= scale, c1.y *= scale;
      const float2 x0 = *reinterpret_cast<const float2*>(r0 + i);
      const float2 y0 = *reinterpret_cast<const float2*>(r0 + i + HALF);
      const float2 x1 = *reinterpret_cast<const float2*>(r1 + i);
      const float2 y1 = *reinterpret_cast<const float2*>(r1 + i + HALF);
      xr[0][2 * e2] = fmaf(x0.x, c0.x, -y0.x * c0.y);
      xr[0][2 * e2 + 1] = fmaf(x0.y, c1.x, -y0.y * c1.y);
      yr[0][2 * e2] = fmaf(y0.x, c0.x, x0.x * c0.y);
      yr[0][2 * e2 + 1] = fmaf(y0.y, c1.x, x0.y * c1.y);
      xr[1][2 * e2] = fmaf(x1.x, c0.x, -y1.x * c0.y);
      xr[1][2 * e2 + 1] = fmaf(x1.y, c1.x, -y1.y * c1.y);
      yr[1][2 * e2] = fmaf(y1.x, c0.x, x1.x * c0.y);
      yr[1][2 * e2 + 1] = fmaf(y1.y, c1.x, x1.y * c1.y);
    }
    qa[ks][0] = pack_op2<F16>(xr[0][0], xr[0][1]);
    qa[ks][1] = pack_op2<F16>(xr[1][0], xr[1][1]);
    qa[ks][2] = pack_op2<F16>(xr[0][2], xr[0][3]);
    qa[ks][3] = pack_op2<F16>(xr[1][2], xr[1][3]);
    qa[ks + D / 32][0] = pack_op2<F16>(yr[0][0], yr[0][1]);
    qa[ks + D / 32][1] = pack_op2<F16>(yr[1][0], yr[1][1]);
    qa[ks + D / 32][2] = pack_op2<F16>(yr[0][2], yr[0][3]);
    qa[ks + D / 32][3] = pack_op2<F16>(yr[1][2], yr[1][3]);
  }
}

// ALIBI (with LAZY = false, key-position words): q is built once (the caller's table
// has zero rates: no rotation), and every score of row r gets slope_r (n - m) in log2
// units, n = the block word's position + slot, m = q_pos.
// f16 A fragments of scale * R_delta q (D = 128) in the permuted head-dimension order
// of the FP8 decode's K fragments: k-step ks, columns 2t + {0,1} and 2t + 8 + {0,1}
// hold dimensions 32t + 4ks + {0,1} and {2,3} (t = lane & 3), so lanes t = 0, 1 hold
// first halves of rotate-half pairs and t = 2, 3 second halves. cs[j] is this lane's
// (cos, sin) of frequency lane + 32 j.
template <int QS_STRIDE>
__device__ __forceinline__ void build_q_frags_perm(uint32_t (&qa)[8][4], const float* __restrict__ qs, int mt,
                                                   int lane, float scale, const float2 (&cs)[2]) {
  const int g = lane >> 2, t = lane & 3;
  const bool second = t >= 2;
  const float* r0 = qs + (mt * 16 + g) * QS_STRIDE;
  const float* r1 = r0 + 8 * QS_STRIDE;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    float v0[4], v1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 4 * ks + e;
      const int d = 32 * t + i, dp = second ? d - 64 : d + 64;  // own dimension and its pair partner
      // frequency d mod 64 = 32 (t & 1) + i: lane i's cs[t & 1]
      const float2 ca = make_float2(__shfl_sync(0xffffffffu, cs[0].x, i), __shfl_sync(0xffffffffu, cs[0].y, i));
      const float2 cb = make_float2(__shfl_sync(0xffffffffu, cs[1].x, i), __shfl_sync(0xffffffffu, cs[1].y, i));
      const float c = ((t & 1) ? cb.x : ca.x) * scale;
      const float sn = ((t & 1) ? cb.y : ca.y) * scale;
      // first half: x c - y s; second half: y c + x s (own value times c, partner times s)
      v0[e] = fmaf(r0[d], c, (second ? r0[dp] : -r0[dp]) * sn);
      v1[e] = fmaf(r1[d], c, (second ? r1[dp] : -r1[dp]) * sn);
    }
    qa[ks][0] = pack_f16x2(v0[0], v0[1]);
    qa[ks][1] = pack_f16x2(v1[0], v1[1]);
    qa[ks][2] = pack_f16x2(v0[2], v0[3]);
    qa[ks][3] = pack_f16x2(v1[2], v1[3]);
  }
}

// FP8 (D = 128): the pools hold e4m3 codes. Each block lands in the ring as codes,
// the team converts it (exactly) to f16 in its conversion buffer, and the block is
// attended with f16 operands, scores scaled by k_scale; the output is scaled by
// v_scale.
template <int D, int MT, int SPT, bool LAZY, bool ALIBI = false, bool FP8 = false>
__global__ void __launch_bounds__(DecodeCfg<D, MT, SPT>::NTHREADS, MT == 1 ? 3 : 1)
    decode_bf16_kernel(const std::conditional_t<ALIBI, DecodeAlibiArgs,
                                                std::conditional_t<FP8, DecodeFp8Args, DecodeArgs>> a,
                       const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  static_assert(!(ALIBI && LAZY), "the ALiBi variant does not rotate");
  static_assert(!(ALIBI && FP8) && (!FP8 || D == 128), "FP8 KV: d = 128, no ALiBi");
  using C = DecodeCfg<D, MT, SPT, FP8>;
  constexpr int HALF = C::HALF, CPL = (HALF + 31) / 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = align1024(smem_raw);
  float* qs = reinterpret_cast<float*>(stages + C::STAGES_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::STAGES_BYTES + C::QS_BYTES);
  __shared__ int abort_flag;

  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int team = warp / MT, mt = warp % MT;
  const int g = lane >> 2, t = lane & 3;
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const int b0 = split * a.bps;
  const int n = max(0, min(nb, b0 + a.bps) - b0);
  const int m_pos = a.q_pos[s];
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;

  // Unrotated q of the group, fp32, zero rows past g.
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q) + ((size_t)s * a.Hq + (size_t)kvh * a.G) * D;
  for (int idx = threadIdx.x; idx < C::ROWS * D; idx += C::NTHREADS) {
    const int r = idx / D, c = idx % D;
    qs[r * C::QS_STRIDE + c] = r < a.G ? __bfloat162float(qg[idx]) : 0.f;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::TEAMS * SPT; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ team setup
  // Team t owns a contiguous quarter of the split, so a warp meets only the
  // document boundaries inside its own range (each costs a q re-rotation).
  const int per_team = (n + C::TEAMS - 1) / C::TEAMS;
  const int kb0 = team * per_team;
  const int nk = max(0, min(n, kb0 + per_team) - kb0);  // blocks of this team
  uint8_t* tst = stages + team * C::TEAM_BYTES;
  const uint32_t conv = smem_u32(tst + SPT * C::STAGE_BYTES);  // FP8: the f16 tile buffer
  uint64_t* tfull = full + team * SPT;
  const bool leader = (mt == 0 && lane == 0);
  auto issue_load = [&](uint8_t* stage, uint64_t* bar, int phys) {
    if constexpr (FP8) load_block_fp8(stage, bar, phys, a.num_pool_blocks, a.Hkv, kvh, &kmap, &vmap);
    else load_block<D>(stage, bar, phys, a.num_pool_blocks, a.Hkv, kvh, &kmap, &vmap);
  };
  auto block_of = [&](int k) { return b0 + kb0 + k; };
  auto load_words = [&](int kc, uint32_t& w, uint32_t& wn) {
    const int k = kc + lane, b = block_of(k);
    w = k < nk ? __ldg(&wrow[b]) : 0u;
    wn = (k < nk && b + 1 < nb) ? __ldg(&wrow[b + 1]) : 0u;
  };
  auto describe = [&](int kc, uint32_t w, uint32_t wn) {
    const int k = kc + lane;
    return describe_block(k < nk, block_of(k), nb, seq_len, w, wn, a.id_bits, a.num_pool_blocks, a.status);
  };
  uint32_t w_cur, wn_cur, w_nxt = 0, wn_nxt = 0;
  load_words(0, w_cur, wn_cur);
  if (nk > 32) load_words(32, w_nxt, wn_nxt);
  LaneBlock cur = describe(0, w_cur, wn_cur), nxt{a.num_pool_blocks, 0, 0};
  bool nxt_ready = false;
  int issued = 0;
  {
    const int pro = min(SPT, nk);
    for (int k = 0; k < pro; ++k) {
      const int phys = __shfl_sync(0xffffffffu, cur.phys, k);
      if (leader) issue_load(tst + k * C::STAGE_BYTES, &tfull[k], phys);
    }
    issued = pro;
  }

  // ------------------------------------------------------------ q fragments
  uint32_t qa[D / 16][4];
  float2 tr[CPL], cs[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) tr[j] = __ldg(&a.rope[lane + 32 * j]);
  // Each lane evaluates cos/sin for frequencies lane + 32 j; fragments gather them by shuffle.
  auto rebuild = [&](int delta) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) cs[j] = rope_cs(tr[j], delta, a.status);
    if constexpr (FP8) {
      build_q_frags_perm<C::QS_STRIDE>(qa, qs, mt, lane, a.scale_log2, cs);
    } else {
      build_q_frags<D, C::QS_STRIDE>(qa, qs, mt, lane, a.scale_log2, [&](int ks, int i) {
        const float2 v = cs[(16 * ks) >> 5];
        return make_float2(__shfl_sync(0xffffffffu, v.x, i & 31), __shfl_sync(0xffffffffu, v.y, i & 31));
      });
    }
  };
  if constexpr (!LAZY) rebuild(m_pos);  // control: pool holds absolute-position keys, rotate q once by R_m
  float ab_slope[2] = {0.f, 0.f};
  if constexpr (ALIBI) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = mt * 16 + g + 8 * rr;
      if (row < a.G) ab_slope[rr] = __ldg(&a.alibi[kvh * a.G + row]) * 1.4426950408889634f;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const LdsmLane ln = ldsm_lane(lane);
  int k = 0, cbase = 0;  // next block of the team; first block of the current word chunk
  int p_seg = nk > 0 ? __shfl_sync(0xffffffffu, cur.p, 0) : 0;
  bool aborted = false;
  // Outer loop: one pass per document run of the team's range (lazy only; the
  // control runs it once). The q re-rotation sits here, outside the per-block
  // loop, and overlaps the loads already in flight for the run's first block.
  while (k < nk && !aborted) {
    if constexpr (LAZY) rebuild(m_pos - p_seg);
  for (; k < nk; ++k) {
    if (k - cbase >= 32) {  // advance the word chunk
      if (!nxt_ready) nxt = describe(k, w_nxt, wn_nxt);
      cur = nxt;
      nxt_ready = false;
      cbase += 32;
      if (k + 32 < nk) load_words(k + 32, w_nxt, wn_nxt);
    }
    const int slot = k % SPT;
    const int nvalid = __shfl_sync(0xffffffffu, cur.nv, k & 31);
    if constexpr (LAZY) {
      const int p = __shfl_sync(0xffffffffu, cur.p, k & 31);
      if (p != p_seg) {  // next document: leave to re-rotate q, then resume at block k
        p_seg = p;
        break;
      }
    }
    bool ok = warp_wait(&tfull[slot], (k / SPT) & 1, a.status);
    if constexpr (ALIBI) {
      const int pk = __shfl_sync(0xffffffffu, cur.p, k & 31);  // this block's first key position
      const float b0[2] = {ab_slope[0] * (float)(pk - m_pos), ab_slope[1] * (float)(pk - m_pos)};
      if (ok) attend_block_bias<D>(smem_u32(tst + slot * C::STAGE_BYTES), ln, qa, nvalid, o, m_r, l_r, lane, b0, ab_slope);
    } else if constexpr (FP8) {
      if (ok) convert_fp8_block(tst + slot * C::STAGE_BYTES, tst + SPT * C::STAGE_BYTES, 32 * mt + lane, 32 * MT);
      // the team's f16 tiles are complete before any warp reads them
      if constexpr (MT > 1) ok = team_and(team, 32 * MT, ok);
      else __syncwarp();
      if constexpr (FP8) {  // always true here; keeps the D = 128 call out of other instantiations
        if (ok)
          attend_block_fp8(smem_u32(tst + slot * C::STAGE_BYTES), conv, ln, qa, nvalid, o, m_r, l_r, lane,
                           a.k_scale);
      }
    } else {
      if (ok) attend_block<D>(smem_u32(tst + slot * C::STAGE_BYTES), ln, qa, nvalid, o, m_r, l_r, lane);
    }
    // The team's warps are all done with this stage (and agree to go on) before it is refilled.
    if constexpr (MT > 1) ok = team_and(team, 32 * MT, ok);
    if (!ok) {
      abort_flag = 1;
      aborted = true;
      break;
    }
    __syncwarp();
    // Refill this stage with the team's block SPT positions ahead.
    const int kn = k + SPT;
    if (kn < nk) {
      int phys;
      if ((kn >> 5) == (k >> 5)) {
        phys = __shfl_sync(0xffffffffu, cur.phys, kn & 31);
      } else {
        if (!nxt_ready) {
          nxt = describe(kn & ~31, w_nxt, wn_nxt);
          nxt_ready = true;
        }
        phys = __shfl_sync(0xffffffffu, nxt.phys, kn & 31);
      }
      if (leader) issue_load(tst + slot * C::STAGE_BYTES, &tfull[slot], phys);
      issued = kn + 1;
    }
  }
  }
  // Copies still in flight (only after a timeout) must land before exit (bounded).
  if (leader)
    for (int kk = k; kk < issued; ++kk) mbar_wait(&tfull[kk % SPT], (kk / SPT) & 1, a.status);
  // Finish the per-row denominators (the 4 lanes of a quad hold partial sums).
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 1);
    l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 2);
  }
  // Every team is done with its ring: reuse the stages for the team merge.
  __syncthreads();
  if (!abort_flag) {
    float* red = reinterpret_cast<float*>(stages);  // [TEAMS][ROWS][D + 2]
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = mt * 16 + g + 8 * rr;
      if (row < a.G) {
        float* dst = red + ((size_t)team * C::ROWS + row) * (D + 2);
        float vs = 1.f;
        if constexpr (FP8) vs = a.v_scale;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          dst[8 * j + 2 * t] = o[j][2 * rr] * vs;
          dst[8 * j + 2 * t + 1] = o[j][2 * rr + 1] * vs;
        }
        if (t == 0) {
          dst[D] = m_r[rr];
          dst[D + 1] = l_r[rr];
        }
      }
    }
  }
  __syncthreads();
  if (!abort_flag) {
    const float* red = reinterpret_cast<const float*>(stages);
    for (int idx = threadIdx.x; idx < a.G * D; idx += C::NTHREADS) {
      const int row = idx / D, col = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int tm = 0; tm < C::TEAMS; ++tm) M = fmaxf(M, red[((size_t)tm * C::ROWS + row) * (D + 2) + D]);
      float acc = 0.f, L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int tm = 0; tm < C::TEAMS; ++tm) {
          const float* src = red + ((size_t)tm * C::ROWS + row) * (D + 2);
          const float w = exp2f(src[D] - M);
          acc += w * src[col];
          L += w * src[D + 1];
        }
      }
      const int h = kvh * a.G + row;
      if (a.splits == 1) {
        static_cast<__nv_bfloat16*>(a.out)[((size_t)s * a.Hq + h) * D + col] =
            __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
      } else {
        const size_t pidx = ((size_t)s * a.Hq + h) * a.splits + split;
        a.ws_o[pidx * D + col] = acc;
        if (col == 0) {
          a.ws_ml[2 * pidx] = M;
          a.ws_ml[2 * pidx + 1] = L;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ split combine
// out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the splits that hold
// blocks of the sequence (the same rescale as the online softmax).
template <int D, typename T>
__global__ void decode_combine_kernel(const DecodeArgs a) {
  const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= a.B * a.Hq) return;
  const int s = warp_global / a.Hq;
  int seq_len = a.seq_lens[s];
  seq_len = seq_len < 0 ? 0 : min(seq_len, kBlock * a.max_blocks);
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const int ns = min(a.splits, (nb + a.bps - 1) / a.bps);
  const size_t base = (size_t)warp_global * a.splits;
  float M = -INFINITY;
  for (int sp = lane; sp < ns; sp += 32) M = fmaxf(M, a.ws_ml[2 * (base + sp)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int sp = 0; sp < ns; ++sp) {
      const float m = a.ws_ml[2 * (base + sp)];
      const float w = exp2f(m - M);  // empty split: m = -inf -> w = 0
      L += w * a.ws_ml[2 * (base + sp) + 1];
      const float* src = a.ws_o + (base + sp) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x, acc[1] += w * v.y, acc[2] += w * v.z, acc[3] += w * v.w;
      } else {
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] += w * src[j];
      }
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  T* dst = static_cast<T*>(a.out) + (size_t)warp_global * D + lane * PER;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    if constexpr (sizeof(T) == 2)
      dst[j] = __float2bfloat16_rn(acc[j] * inv);
    else
      dst[j] = acc[j] * inv;
  }
}

// ------------------------------------------------------------------ debug gather
// Same word decode, hole rule and TMA box loads as decode, in a plain
// producer/consumer pair: warp 0 loads, warp 1 copies each block out of the
// swizzled stage into a dense buffer.
template <int D>
__global__ void __launch_bounds__(64) gather_bf16_kernel(const GatherArgs a, const __grid_constant__ CUtensorMap kmap,
                                                         const __grid_constant__ CUtensorMap vmap) {
  constexpr int NS = 4, NBOX = D / 64, BOX_BYTES = kBlock * 128, KV_BYTES = NBOX * BOX_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = align1024(smem_raw);
  int* meta = reinterpret_cast<int*>(stages + NS * 2 * KV_BYTES);  // [NS][2]: p, nvalid
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + 2 * NS);
  uint64_t* empty = full + NS;
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const size_t rows = (size_t)kBlock * a.max_blocks;
  __nv_bfloat16* kout = static_cast<__nv_bfloat16*>(a.k_out) + ((size_t)s * a.Hkv + kvh) * rows * D;
  __nv_bfloat16* vout = static_cast<__nv_bfloat16*>(a.v_out) + ((size_t)s * a.Hkv + kvh) * rows * D;
  if (warp == 0) {
    int issued = 0;
    bool ok = true;
    for (int c0 = 0; c0 < nb && ok; c0 += 32) {
      const int b = c0 + lane;
      const uint32_t w = b < nb ? __ldg(&wrow[b]) : 0u;
      const uint32_t wn = b + 1 < nb ? __ldg(&wrow[b + 1]) : 0u;
      const LaneBlock lb = describe_block(b < nb, b, nb, seq_len, w, wn, a.id_bits, a.num_pool_blocks, a.status);
      for (int j = 0; j < min(32, nb - c0); ++j) {
        const int i = c0 + j, st = i % NS;
        const int phys = __shfl_sync(0xffffffffu, lb.phys, j);
        const int p = __shfl_sync(0xffffffffu, lb.p, j);
        const int nv = __shfl_sync(0xffffffffu, lb.nv, j);
        if (i >= NS && !warp_wait(&empty[st], ((i / NS) & 1) ^ 1, a.status, a.wait_ns)) {
          ok = false;
          break;
        }
        // A withheld block (failure-path test) gets neither its copies nor the arrival
        // that expects them: its stage's phase never completes and no copy is in flight.
        const bool withhold = i == a.withhold_block && s == 0 && kvh == 0;
        if (lane == 0 && !withhold) {
          meta[2 * st] = p;
          meta[2 * st + 1] = nv;
          load_block<D>(stages + st * 2 * KV_BYTES, &full[st], phys, a.num_pool_blocks, a.Hkv, kvh, &kmap, &vmap);
        }
        issued = i + 1;
      }
    }
    if (lane == 0)
      for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(&full[i % NS], (i / NS) & 1, a.status, a.wait_ns);
  } else {
    for (int i = 0; i < nb; ++i) {
      const int st = i % NS;
      if (!warp_wait(&full[st], (i / NS) & 1, a.status, a.wait_ns)) break;
      const int p = meta[2 * st], nvalid = meta[2 * st + 1];
      const uint8_t* kb = stages + st * 2 * KV_BYTES;
      const uint8_t* vb = kb + KV_BYTES;
      for (int idx = lane; idx < kBlock * (D / 8); idx += 32) {
        const int row = idx / (D / 8), chunk = idx % (D / 8);
        const uint32_t off = (chunk >> 3) * BOX_BYTES + sw128(row, chunk & 7);
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (row < nvalid) {
          kv = *reinterpret_cast<const uint4*>(kb + off);
          vv = *reinterpret_cast<const uint4*>(vb + off);
        }
        const size_t o = ((size_t)kBlock * i + row) * D + chunk * 8;
        *reinterpret_cast<uint4*>(kout + o) = kv;
        *reinterpret_cast<uint4*>(vout + o) = vv;
      }
      if (a.pos_out && kvh == 0 && lane < kBlock)
        a.pos_out[(size_t)s * rows + kBlock * i + lane] = lane < nvalid ? p : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // Rows past the sequence: zero / -1.
    for (size_t idx = (size_t)kBlock * nb * (D / 8) + lane; idx < rows * (D / 8); idx += 32) {
      *reinterpret_cast<uint4*>(kout + idx * 8) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(vout + idx * 8) = make_uint4(0, 0, 0, 0);
    }
    if (a.pos_out && kvh == 0)
      for (size_t r = (size_t)kBlock * nb + lane; r < rows; r += 32) a.pos_out[(size_t)s * rows + r] = -1;
  }
}

// ------------------------------------------------------------------ launchers

template <int D, int MT, bool LAZY, bool ALIBI, bool FP8 = false>
static cudaError_t launch_decode_t(const DecodeArgs& a, const float* alibi, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, cudaStream_t st, float k_scale = 1.f,
                                   float v_scale = 1.f) {
  constexpr int SPT = LAZY_DECODE_SPT;
  using C = DecodeCfg<D, MT, SPT, FP8>;
  auto kern = decode_bf16_kernel<D, MT, SPT, LAZY, ALIBI, FP8>;
  cudaError_t e = set_smem_once<decode_bf16_kernel<D, MT, SPT, LAZY, ALIBI, FP8>>(C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.B);
  if constexpr (FP8) {
    (void)alibi;
    DecodeFp8Args fa;
    static_cast<DecodeArgs&>(fa) = a;
    fa.k_scale = k_scale;
    fa.v_scale = v_scale;
    kern<<<grid, C::NTHREADS, C::SMEM, st>>>(fa, kmap, vmap);
  } else if constexpr (ALIBI) {
    DecodeAlibiArgs aa;
    static_cast<DecodeArgs&>(aa) = a;
    aa.alibi = alibi;
    kern<<<grid, C::NTHREADS, C::SMEM, st>>>(aa, kmap, vmap);
  } else {
    (void)alibi;
    kern<<<grid, C::NTHREADS, C::SMEM, st>>>(a, kmap, vmap);
  }
  return cudaGetLastError();
}

template <int D, bool LAZY, bool ALIBI>
static cudaError_t dispatch_mt(const DecodeArgs& a, const float* alibi, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t st) {
  if (a.G <= 16) return launch_decode_t<D, 1, LAZY, ALIBI>(a, alibi, kmap, vmap, st);
  if (a.G <= 32) return launch_decode_t<D, 2, LAZY, ALIBI>(a, alibi, kmap, vmap, st);
  return launch_decode_t<D, 4, LAZY, ALIBI>(a, alibi, kmap, vmap, st);
}

int decode_bf16_smem_bytes(int D, int G) {
  constexpr int S = LAZY_DECODE_SPT;
  if (D == 64)
    return G <= 16 ? DecodeCfg<64, 1, S>::SMEM : G <= 32 ? DecodeCfg<64, 2, S>::SMEM : DecodeCfg<64, 4, S>::SMEM;
  return G <= 16 ? DecodeCfg<128, 1, S>::SMEM : G <= 32 ? DecodeCfg<128, 2, S>::SMEM : DecodeCfg<128, 4, S>::SMEM;
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, const float* alibi, bool lazy, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t st) {
  if (alibi)
    return a.D == 128 ? dispatch_mt<128, false, true>(a, alibi, kmap, vmap, st)
                      : dispatch_mt<64, false, true>(a, alibi, kmap, vmap, st);
  if (a.D == 128)
    return lazy ? dispatch_mt<128, true, false>(a, nullptr, kmap, vmap, st)
                : dispatch_mt<128, false, false>(a, nullptr, kmap, vmap, st);
  return lazy ? dispatch_mt<64, true, false>(a, nullptr, kmap, vmap, st)
              : dispatch_mt<64, false, false>(a, nullptr, kmap, vmap, st);
}

template <bool LAZY>
static cudaError_t dispatch_fp8(const DecodeArgs& a, float ks, float vs, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t st) {
  if (a.G <= 16) return launch_decode_t<128, 1, LAZY, false, true>(a, nullptr, kmap, vmap, st, ks, vs);
  if (a.G <= 32) return launch_decode_t<128, 2, LAZY, false, true>(a, nullptr, kmap, vmap, st, ks, vs);
  return launch_decode_t<128, 4, LAZY, false, true>(a, nullptr, kmap, vmap, st, ks, vs);
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, float k_scale, float v_scale, bool lazy, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t st) {
  if (a.D != 128) return cudaErrorInvalidValue;
  return lazy ? dispatch_fp8<true>(a, k_scale, v_scale, kmap, vmap, st)
              : dispatch_fp8<false>(a, k_scale, v_scale, kmap, vmap, st);
}

cudaError_t launch_combine(const DecodeArgs& a, bool out_bf16, cudaStream_t st) {
  const int warps = a.B * a.Hq;
  if (warps == 0) return cudaSuccess;
  const int threads = 256, blocks = (warps + 7) / 8;
  if (a.D == 128) {
    if (out_bf16)
      decode_combine_kernel<128, __nv_bfloat16><<<blocks, threads, 0, st>>>(a);
    else
      decode_combine_kernel<128, float><<<blocks, threads, 0, st>>>(a);
  } else {
    if (out_bf16)
      decode_combine_kernel<64, __nv_bfloat16><<<blocks, threads, 0, st>>>(a);
    else
      decode_combine_kernel<64, float><<<blocks, threads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_bf16(const GatherArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  dim3 grid(a.Hkv, a.B);
  const int smem = 1024 + 4 * 2 * (a.D / 64) * kBlock * 128 + 4 * 2 * 4 + 2 * 4 * 8;
  if (a.D == 128) {
    cudaError_t e = cudaFuncSetAttribute(gather_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gather_bf16_kernel<128><<<grid, 64, smem, st>>>(a, kmap, vmap);
  } else {
    cudaError_t e = cudaFuncSetAttribute(gather_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gather_bf16_kernel<64><<<grid, 64, smem, st>>>(a, kmap, vmap);
  }
  return cudaGetLastError();
}

}  // namespace lazy
