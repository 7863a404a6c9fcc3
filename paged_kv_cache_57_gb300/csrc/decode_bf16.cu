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
// is what turns the 16-token block into a small dense contraction):
//
//   producer warp : per logical block, decodes the word (phys id, document start
//                   p, valid slots), stages cos/sin of (m - p) for every
//                   frequency, and TMA-loads the 16 x d K and V rows of the
//                   block (128-byte swizzled boxes) into a ring of NS stages
//                   guarded by full/empty mbarriers.
//   consumer teams: TEAMS teams of MT warps; team t takes blocks t, t+TEAMS, ...
//                   Each warp keeps the A fragments of R_{m-p} q for its 16 rows
//                   and rebuilds them only when p changes; S = q' K^T and
//                   O += P V run on mma.sync (bf16 in, fp32 accumulate) with an
//                   online (max, sum) softmax ("KV Cache, Flash Attention &
//                   Otimização de Inferência", "Flash Attention -- tiling").
//   merge         : teams combine in shared memory with the same max/sum
//                   rescale; a split writes fp32 partials (or, with one split,
//                   the final output) and decode_combine merges the splits.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace lazy {

template <int HALF>
struct __align__(16) StageMeta {
  int p;       // document start position of the block
  int nvalid;  // valid slots (0..16); 0 also for a skipped (invalid) block
  int pad[2];
  float2 cs[HALF];  // (cos, sin) of (m - p) * w_i
};

template <int D, int MT>
struct DecodeCfg {
  static constexpr int TEAMS = (MT >= 4) ? 2 : 4;
  static constexpr int CW = TEAMS * MT;  // consumer warps
  static constexpr int NTHREADS = 32 * (CW + 1);
  static constexpr int HALF = D / 2;
  static constexpr int NBOX = D / 64;  // 64-column (128-byte) TMA boxes per row
  static constexpr int BOX_BYTES = kBlock * 128;
  static constexpr int KV_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int ROWS = MT * 16;
  static constexpr int MERGE_BYTES = TEAMS * ROWS * (D + 2) * 4;
  static constexpr int NS_MIN = (MERGE_BYTES + STAGE_BYTES - 1) / STAGE_BYTES;
  static constexpr int NS = ((NS_MIN > 8 ? NS_MIN : 8) + TEAMS - 1) / TEAMS * TEAMS;
  static constexpr int STAGES_BYTES = NS * STAGE_BYTES;
  static constexpr int META_BYTES = NS * (int)sizeof(StageMeta<HALF>);
  static constexpr int QS_BYTES = ROWS * D * 4;
  static constexpr int BAR_BYTES = 2 * NS * 8;
  static constexpr int SMEM = 1024 + STAGES_BYTES + META_BYTES + QS_BYTES + BAR_BYTES;
  static constexpr int CS_PER_LANE = HALF / 32;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait: every lane polls, and the warp gives up together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

// The producer warp of a split: blocks b0 .. b0+n-1 of one sequence. Words are
// fetched 32 at a time (one per lane) one chunk ahead, so no word load sits on
// the issue path. Per block: wait for the stage to be free, write the stage's
// metadata (document start p, valid slots, and cos/sin of (m - p) when the
// document changes -- computed in registers, no memory access), then lane 0
// arms the full barrier and issues the TMA loads of the block's K and V rows.
// Invalid block ids are not loaded: the stage is marked empty (nvalid = 0).
// Returns the number of blocks issued (all of them unless a wait timed out).
template <int D, bool WITH_CS, int NS, int STAGE_BYTES>
__device__ __forceinline__ int producer_loop(int lane, int b0, int n, int nb, int seq_len,
                                             const uint32_t* __restrict__ wrow, int id_bits, int num_pool_blocks,
                                             int hkv, int kvh, StageMeta<D / 2>* meta, uint8_t* stages,
                                             uint64_t* full, uint64_t* empty, const CUtensorMap* kmap,
                                             const CUtensorMap* vmap, int m_pos, const float2* __restrict__ turns,
                                             unsigned int* status) {
  constexpr int HALF = D / 2, CPL = HALF / 32, NBOX = D / 64, BOX_BYTES = kBlock * 128;
  float2 tr[CPL], cs[CPL];
  if constexpr (WITH_CS) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) tr[j] = __ldg(&turns[lane + 32 * j]);
  }
  int p_cur = INT_MIN;
  auto load_chunk = [&](int c0, uint32_t& w, uint32_t& wn) {
    const int r = c0 + lane, b = b0 + r;
    w = r < n ? __ldg(&wrow[b]) : 0u;
    wn = (r < n && b + 1 < nb) ? __ldg(&wrow[b + 1]) : 0u;
  };
  uint32_t wa = 0, wna = 0, wb = 0, wnb = 0;
  load_chunk(0, wa, wna);
  int issued = 0;
  for (int c0 = 0; c0 < n; c0 += 32) {
    if (c0 + 32 < n) load_chunk(c0 + 32, wb, wnb);
    const int r = c0 + lane, b = b0 + r;
    const BlockInfo bi = decode_word(wa, b, id_bits);
    const int pn = (b + 1 < nb) ? decode_word(wna, b + 1, id_bits).p : bi.p;
    int nv = block_valid(b, nb, seq_len, bi.p, pn);
    nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
    if (bi.phys >= num_pool_blocks) {
      nv = 0;
      if (r < n) raise_status(status, LAZY_DEV_BAD_BLOCK_ID);
    }
    const int cnt = min(32, n - c0);
    for (int j = 0; j < cnt; ++j) {
      const int i = c0 + j, st = i % NS;
      const int phys = __shfl_sync(0xffffffffu, bi.phys, j);
      const int p = __shfl_sync(0xffffffffu, bi.p, j);
      const int nvalid = __shfl_sync(0xffffffffu, nv, j);
      if (i >= NS && !warp_wait(&empty[st], ((i / NS) & 1) ^ 1, status)) return issued;
      StageMeta<HALF>* m = &meta[st];
      if constexpr (WITH_CS) {
        if (p != p_cur) {
#pragma unroll
          for (int jj = 0; jj < CPL; ++jj) cs[jj] = rope_cs(tr[jj], m_pos - p, status);
          p_cur = p;
        }
#pragma unroll
        for (int jj = 0; jj < CPL; ++jj) m->cs[lane + 32 * jj] = cs[jj];
      }
      if (lane == 0) {
        m->p = p;
        m->nvalid = nvalid;
      }
      __syncwarp();
      if (lane == 0) {
        uint64_t* fb = &full[st];
        uint8_t* stage = stages + st * STAGE_BYTES;
        if (phys < num_pool_blocks) {
          mbar_arrive_expect_tx(fb, 2 * NBOX * BOX_BYTES);
          const int y = (phys * hkv + kvh) * kBlock;
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx) tma_load_2d(stage + bx * BOX_BYTES, kmap, fb, bx * 64, y);
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx) tma_load_2d(stage + (NBOX + bx) * BOX_BYTES, vmap, fb, bx * 64, y);
        } else {
          mbar_arrive(fb);
        }
      }
      issued = i + 1;
    }
    wa = wb;
    wna = wnb;
  }
  return issued;
}

// Bounded wait, by lane 0, for every copy this CTA still has in flight.
template <int NS>
__device__ __forceinline__ void drain_copies(int lane, int issued, uint64_t* full, unsigned int* status) {
  if (lane == 0)
    for (int i = max(0, issued - NS); i < issued; ++i) mbar_wait(&full[i % NS], (i / NS) & 1, status);
}

// A fragments of R_delta q for rows (mt*16 + g, mt*16 + g + 8), g = lane/4.
// The thread owns columns 16ks + 2t + {0,1,8,9}; ks and ks + D/32 hold the two
// halves of the same rotate-half pairs, so each pair is rotated by one thread.
template <int D, typename CsFn>
__device__ __forceinline__ void build_q_frags(uint32_t (&qa)[D / 16][4], const float* __restrict__ qs, int mt,
                                              int lane, CsFn cs_of) {
  constexpr int HALF = D / 2;
  const int g = lane >> 2, t = lane & 3;
  const float* r0 = qs + (mt * 16 + g) * D;
  const float* r1 = r0 + 8 * D;
#pragma unroll
  for (int ks = 0; ks < D / 32; ++ks) {
    float xr[2][4], yr[2][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 16 * ks + 2 * t + (e & 1) + (e >> 1) * 8;
      const float2 c = cs_of(i);
      const float x0 = r0[i], y0 = r0[i + HALF], x1 = r1[i], y1 = r1[i + HALF];
      xr[0][e] = fmaf(x0, c.x, -y0 * c.y);
      yr[0][e] = fmaf(y0, c.x, x0 * c.y);
      xr[1][e] = fmaf(x1, c.x, -y1 * c.y);
      yr[1][e] = fmaf(y1, c.x, x1 * c.y);
    }
    qa[ks][0] = pack_bf16x2(xr[0][0], xr[0][1]);
    qa[ks][1] = pack_bf16x2(xr[1][0], xr[1][1]);
    qa[ks][2] = pack_bf16x2(xr[0][2], xr[0][3]);
    qa[ks][3] = pack_bf16x2(xr[1][2], xr[1][3]);
    qa[ks + D / 32][0] = pack_bf16x2(yr[0][0], yr[0][1]);
    qa[ks + D / 32][1] = pack_bf16x2(yr[1][0], yr[1][1]);
    qa[ks + D / 32][2] = pack_bf16x2(yr[0][2], yr[0][3]);
    qa[ks + D / 32][3] = pack_bf16x2(yr[1][2], yr[1][3]);
  }
}

template <int D, int MT, bool LAZY>
__global__ void __launch_bounds__(DecodeCfg<D, MT>::NTHREADS)
    decode_bf16_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  using C = DecodeCfg<D, MT>;
  using Meta = StageMeta<C::HALF>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = align1024(smem_raw);
  Meta* meta = reinterpret_cast<Meta*>(stages + C::STAGES_BYTES);
  float* qs = reinterpret_cast<float*>(stages + C::STAGES_BYTES + C::META_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::STAGES_BYTES + C::META_BYTES + C::QS_BYTES);
  uint64_t* empty = full + C::NS;
  __shared__ int abort_flag;

  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    const int r = idx / D;
    qs[idx] = r < a.G ? __bfloat162float(qg[idx]) : 0.f;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MT);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == C::CW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
    }
    const int issued = producer_loop<D, LAZY, C::NS, C::STAGE_BYTES>(
        lane, b0, n, nb, seq_len, wrow, a.id_bits, a.num_pool_blocks, a.Hkv, kvh, meta, stages, full, empty, &kmap,
        &vmap, m_pos, a.rope, a.status);
    if (issued < n) abort_flag = 1;
    drain_copies<C::NS>(lane, issued, full, a.status);
  } else {
    // ------------------------------------------------------------ consumers
    const int team = warp / MT, mt = warp % MT;
    const int g = lane >> 2, t = lane & 3;
    uint32_t qa[D / 16][4];
    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    int p_prev = INT_MIN;
    if constexpr (!LAZY) {
      // Control: the pool holds absolute-position keys; rotate q once by R_m.
      build_q_frags<D>(qa, qs, mt, lane, [&](int i) { return rope_cs(__ldg(&a.rope[i]), m_pos, a.status); });
    }
    const float sl2 = a.scale_log2;
    for (int i = team; i < n; i += C::TEAMS) {
      const int st = i % C::NS;
      if (!warp_wait(&full[st], (i / C::NS) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      const int p = meta[st].p, nvalid = meta[st].nvalid;
      if constexpr (LAZY) {
        if (p != p_prev) {
          const float2* cs_smem = meta[st].cs;
          build_q_frags<D>(qa, qs, mt, lane, [cs_smem](int i) { return cs_smem[i]; });
          p_prev = p;
        }
      }
      const uint32_t kbase = smem_u32(stages + st * C::STAGE_BYTES);
      const uint32_t vbase = kbase + C::KV_BYTES;

      // S = q' K^T for the 16 keys: two n-tiles of 8 keys.
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mat = lane >> 3;
        const int key = (mat >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int chunk = 2 * ks + (mat & 1);
          uint32_t r[4];
          ldsm_x4(r, kbase + (chunk >> 3) * C::BOX_BYTES + sw128(key, chunk & 7));
          mma_16816(sacc[0], qa[ks], r[0], r[1]);
          mma_16816(sacc[1], qa[ks], r[2], r[3]);
        }
      }
      // Online softmax over this block (rows g and g+8 of the tile).
      uint32_t pa[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = (e >> 1) * 8 + 2 * t + (e & 1);
          const float v = sacc[e >> 1][2 * rr + (e & 1)] * sl2;
          sv[e] = key < nvalid ? v : -INFINITY;
        }
        float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_r[rr], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f(m_r[rr] - m_use);
        m_r[rr] = m_new;
        const uint32_t lo = pack_bf16x2(exp2f(sv[0] - m_use), exp2f(sv[1] - m_use));
        const uint32_t hi = pack_bf16x2(exp2f(sv[2] - m_use), exp2f(sv[3] - m_use));
        pa[rr] = lo;      // keys 2t, 2t+1     (a0 / a1)
        pa[2 + rr] = hi;  // keys 8+2t, 8+2t+1 (a2 / a3)
        const __nv_bfloat162 lb = *reinterpret_cast<const __nv_bfloat162*>(&lo);
        const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi);
        l_r[rr] = l_r[rr] * alpha + (__low2float(lb) + __high2float(lb)) + (__low2float(hb) + __high2float(hb));
        if (alpha != 1.f) {
#pragma unroll
          for (int j = 0; j < D / 8; ++j) {
            o[j][2 * rr] *= alpha;
            o[j][2 * rr + 1] *= alpha;
          }
        }
      }
      // O += P V: V^T fragments via ldmatrix.trans, two d-tiles per load.
      {
        const int mat = lane >> 3;
        const int key = (mat & 1) * 8 + (lane & 7);
        uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
        if (nvalid < kBlock) {  // hole slots may hold anything: zero their V
          const int k0 = 2 * t;
          m0 = (k0 < nvalid ? 0x0000ffffu : 0u) | (k0 + 1 < nvalid ? 0xffff0000u : 0u);
          m1 = (k0 + 8 < nvalid ? 0x0000ffffu : 0u) | (k0 + 9 < nvalid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          const int chunk = 2 * c + (mat >> 1);
          uint32_t r[4];
          ldsm_x4_trans(r, vbase + (chunk >> 3) * C::BOX_BYTES + sw128(key, chunk & 7));
          mma_16816(o[2 * c], pa, r[0] & m0, r[1] & m1);
          mma_16816(o[2 * c + 1], pa, r[2] & m0, r[3] & m1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // Finish the per-row denominators (the 4 lanes of a quad hold partial sums).
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 1);
      l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 2);
    }
    // All consumer warps are done with the stages: reuse them for the team merge.
    asm volatile("bar.sync 1, %0;" ::"r"(C::CW * 32) : "memory");
    if (!abort_flag) {
      float* red = reinterpret_cast<float*>(stages);  // [TEAMS][ROWS][D + 2]
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = mt * 16 + g + 8 * rr;
        if (row < a.G) {
          float* dst = red + ((size_t)team * C::ROWS + row) * (D + 2);
#pragma unroll
          for (int j = 0; j < D / 8; ++j) {
            dst[8 * j + 2 * t] = o[j][2 * rr];
            dst[8 * j + 2 * t + 1] = o[j][2 * rr + 1];
          }
          if (t == 0) {
            dst[D] = m_r[rr];
            dst[D + 1] = l_r[rr];
          }
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(C::CW * 32) : "memory");
    if (!abort_flag) {
      const float* red = reinterpret_cast<const float*>(stages);
      for (int idx = threadIdx.x; idx < a.G * D; idx += C::CW * 32) {
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
// Same word decode, hole rule and TMA path as the decode producer; a consumer
// warp copies each block out of the swizzled stage into a dense buffer.
template <int D>
__global__ void __launch_bounds__(64) gather_bf16_kernel(const GatherArgs a, const __grid_constant__ CUtensorMap kmap,
                                                         const __grid_constant__ CUtensorMap vmap) {
  constexpr int NS = 4, HALF = D / 2, NBOX = D / 64, BOX_BYTES = kBlock * 128, KV_BYTES = NBOX * BOX_BYTES;
  using Meta = StageMeta<HALF>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = align1024(smem_raw);
  Meta* meta = reinterpret_cast<Meta*>(stages + NS * 2 * KV_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + NS);
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
    const int issued = producer_loop<D, false, NS, 2 * KV_BYTES>(lane, 0, nb, nb, seq_len, wrow, a.id_bits,
                                                                 a.num_pool_blocks, a.Hkv, kvh, meta, stages, full,
                                                                 empty, &kmap, &vmap, 0, nullptr, a.status);
    drain_copies<NS>(lane, issued, full, a.status);
  } else {
    for (int i = 0; i < nb; ++i) {
      const int st = i % NS;
      if (!warp_wait(&full[st], (i / NS) & 1, a.status)) break;
      const int p = meta[st].p, nvalid = meta[st].nvalid;
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

template <int D, int MT, bool LAZY>
static cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                   cudaStream_t st) {
  using C = DecodeCfg<D, MT>;
  auto kern = decode_bf16_kernel<D, MT, LAZY>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.B);
  kern<<<grid, C::NTHREADS, C::SMEM, st>>>(a, kmap, vmap);
  return cudaGetLastError();
}

template <int D, bool LAZY>
static cudaError_t dispatch_mt(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t st) {
  if (a.G <= 16) return launch_decode_t<D, 1, LAZY>(a, kmap, vmap, st);
  if (a.G <= 32) return launch_decode_t<D, 2, LAZY>(a, kmap, vmap, st);
  return launch_decode_t<D, 4, LAZY>(a, kmap, vmap, st);
}

int decode_bf16_smem_bytes(int D, int G) {
  if (D == 64) return G <= 16 ? DecodeCfg<64, 1>::SMEM : G <= 32 ? DecodeCfg<64, 2>::SMEM : DecodeCfg<64, 4>::SMEM;
  return G <= 16 ? DecodeCfg<128, 1>::SMEM : G <= 32 ? DecodeCfg<128, 2>::SMEM : DecodeCfg<128, 4>::SMEM;
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, bool lazy, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t st) {
  if (a.D == 128) return lazy ? dispatch_mt<128, true>(a, kmap, vmap, st) : dispatch_mt<128, false>(a, kmap, vmap, st);
  return lazy ? dispatch_mt<64, true>(a, kmap, vmap, st) : dispatch_mt<64, false>(a, kmap, vmap, st);
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
  const int smem = 1024 + 4 * 2 * (a.D / 64) * kBlock * 128 + 4 * (16 + 8 * (a.D / 2)) + 64;
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
