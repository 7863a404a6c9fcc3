// decode_shared.cu -- LazyAttention decode over shared document runs (sm_103a).
//
// The position-agnostic cache ("Resumo Técnico: LazyAttention", "Metodologia:
// Codificação Posicional Diferida") stores each document's K and V once, so a
// batch in which many sequences cite the same documents holds each of those
// blocks once in HBM, at whatever offset each sequence places it. This kernel
// reads each such block once per KV head for the whole batch: a work item is one
// chunk of one document occurrence shared by up to 16 sequences ("members"),
// possibly at 16 different offsets p. Every member gets its own query rotation
// R_{m-p} q ("Implementação Técnica", item 2: the query is rotated by the
// relative offset, only once per document run), and all members' rotated query
// heads become the rows of the mma.sync tiles that consume the block.
//
// CTA: 4 warps. An item has rows = members x g (g = Hq/Hkv query heads per KV
// head), at most 64, i.e. RT = 1, 2 or 4 row tiles of 16. The warps form
// TEAMS = 4/RT teams of RT warps; team t owns a contiguous part of the item's
// blocks and a ring of 8/TEAMS TMA stages (the per-block step, loads and waits
// are those of decode_bf16.cu). Teams merge in shared memory, and every
// (member, query head) writes one fp32 partial (m, l, o) to its slot; the
// combine kernel merges a sequence's slots with the online-softmax rescale.
//
// FP8 (d = 128): the pools hold e4m3 codes (one 16-row x 128-byte box per block for
// K and for V, half the bytes). A team converts each landed V box exactly to f16 in
// its own tile buffer; the K fragments are converted from the codes directly, the
// query fragments are f16 in the permuted head-dimension order of those K fragments,
// scores are scaled by k_scale and the partial outputs by v_scale. (Converting K
// into the team's tile too, once for all of its row tiles, measured slower: the
// tile's stores, barrier and reloads cost more than each warp's own conversion.)
#include <cfloat>
#include <type_traits>

#include "decode_block.cuh"
#include "kernels.h"

namespace lazy {

namespace {

constexpr int kShWarps = 4;
constexpr int kShThreads = 32 * kShWarps;
constexpr int kShRows = 64;    // rows per item at most (4 row tiles)
constexpr int kShStages = 8;   // TMA stages shared out among the teams
constexpr int kShMembers = LAZY_PLAN_MAX_MEMBERS;
constexpr int kItemInts = LAZY_PLAN_ITEM_INTS;  // 8 header ints, 4 per member, then block ids
constexpr int kRecIds = 8 + 4 * kShMembers;      // offset of the block ids in the record
constexpr int kRecBlocks = LAZY_PLAN_ITEM_BLOCK_IDS;
static_assert(kItemInts == kRecIds + kRecBlocks && kItemInts % 4 == 0 && kItemInts / 4 <= kShThreads,
              "item record layout");

template <int D, bool FP8 = false>
struct SharedCfg {
  using G = BlockGeom<D>;
  static constexpr int RED_STRIDE = D + 4;  // merge rows: o[D], m, l, padding to 16 bytes
  static constexpr int STAGE_BYTES = FP8 ? 2 * kBlock * D : G::STAGE_BYTES;  // e4m3: one byte per element
  // e4m3 blocks are half the size: 12 stages (divisible by 1, 2 and 4 teams) keep
  // three quarters of the bytes in flight while three CTAs still fit an SM
  static constexpr int STAGES = FP8 ? 12 : kShStages;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  // FP8: one f16 V tile per team (at most kShWarps teams), the bf16 tile layout
  static constexpr int CONV_BYTES = FP8 ? kShWarps * G::KV_BYTES : 0;
  static constexpr int MERGE_BYTES = kShRows * RED_STRIDE * 4;
  static constexpr int BUF_BYTES =
      ((RING_BYTES + CONV_BYTES > MERGE_BYTES ? RING_BYTES + CONV_BYTES : MERGE_BYTES) + 1023) / 1024 * 1024;
  static constexpr int CS_BYTES = kShMembers * (D / 2) * 8;  // (cos, sin) per member and frequency
  static constexpr int BAR_BYTES = STAGES * 8;
  static constexpr int REC_BYTES = kItemInts * 4;
  static constexpr int META_BYTES = 2 * kShMembers * 4;
  static constexpr int SMEM = 1024 + BUF_BYTES + CS_BYTES + BAR_BYTES + REC_BYTES + META_BYTES;
  static_assert(!FP8 || 3 * SMEM <= 227 * 1024, "three e4m3 CTAs per SM");
};

}  // namespace

// One block's K and V rows of KV head kvh into `stage` (K then V, each as the D/64
// swizzled 64-column boxes attend_block reads), with one 3-D copy each (the map
// views a pool as (column in a 64-column half, row, half)); an id outside the
// pool is not loaded (the barrier is just arrived). No proxy fence is needed
// before the copies: the team's reads of the stage's previous contents have
// returned (their values fed the MMAs) before the team barrier that precedes the
// refill.
template <int D>
__device__ __forceinline__ void load_block_3d(uint8_t* stage, uint64_t* bar, int phys, int num_pool_blocks, int hkv,
                                              int kvh, const CUtensorMap* kmap, const CUtensorMap* vmap) {
  using G = BlockGeom<D>;
  if (phys < num_pool_blocks) {
    mbar_arrive_expect_tx(bar, G::STAGE_BYTES);
    const int y = (phys * hkv + kvh) * kBlock;
    tma_load_3d(stage, kmap, bar, 0, y, 0);
    tma_load_3d(stage + G::KV_BYTES, vmap, bar, 0, y, 0);
  } else {
    mbar_arrive(bar);
  }
}

// Optional per-CTA phase timestamps (build with -DLAZY_DECODE_TRACE): 8 x u64 per
// CTA after the partials in the workspace: start, first loads issued, query
// fragments ready, main loop done, end, (sm id, item), (row tiles, blocks).
#ifdef LAZY_DECODE_TRACE
#define LAZY_TRACE(i, v)                                                                                        \
  do {                                                                                                          \
    if (threadIdx.x == 0)                                                                                       \
      reinterpret_cast<uint64_t*>(a.ws_ml + 2 * (size_t)a.num_slots * a.Hq)[8 * (size_t)blockIdx.x + (i)] = (v); \
  } while (0)
#else
#define LAZY_TRACE(i, v) \
  do {                   \
  } while (0)
#endif

template <int D, bool LAZY, bool ALIBI, bool FP8 = false>
__global__ void __launch_bounds__(kShThreads, 3)
    decode_shared_kernel(const std::conditional_t<ALIBI, SharedAlibiArgs,
                                                  std::conditional_t<FP8, SharedFp8Args, SharedDecodeArgs>> a,
                         const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  static_assert(!FP8 || (D == 128 && !ALIBI), "FP8 KV: d = 128, no ALiBi");
  using C = SharedCfg<D, FP8>;
  using G = BlockGeom<D>;
  constexpr int HALF = D / 2;
  constexpr int NQ = D / 32;  // k-step pairs of a fragment row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align1024(smem_raw);
  float2* cs_tab = reinterpret_cast<float2*>(ring + C::BUF_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::BUF_BYTES + C::CS_BYTES);
  int* rec = reinterpret_cast<int*>(full + C::STAGES);  // the item record
  int* m_delta = rec + kItemInts;                        // rotation offset of each member
  int* m_ok = m_delta + kShMembers;                      // member passed its checks
  __shared__ int abort_flag;

  LAZY_TRACE(0, global_timer_ns());
  // The combine kernel may be scheduled once every CTA of this grid has started;
  // it waits for this grid's completion before it reads the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kvh = blockIdx.x % a.Hkv;
  const int item = blockIdx.x / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ------------------------------------------------------------ item record (one round trip)
  if (threadIdx.x < kItemInts / 4)
    reinterpret_cast<int4*>(rec)[threadIdx.x] =
        __ldg(reinterpret_cast<const int4*>(a.items) + (size_t)item * (kItemInts / 4) + threadIdx.x);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < C::STAGES; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  const int src = rec[0], b0 = rec[1], nblk = rec[2], last_nv = rec[3], nmem = rec[4];
  const bool item_ok = src >= 0 && src < a.B && b0 >= 0 && nblk >= 1 && nblk <= a.max_blocks - b0 &&
                       last_nv >= 1 && last_nv <= kBlock && nmem >= 1 && nmem <= kShMembers &&
                       nmem * a.G <= kShRows;
  if (!item_ok) {  // uniform over the CTA: nothing is loaded or written
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
    return;
  }
  auto mem_seq = [&](int m) { return rec[8 + 4 * m]; };
  auto mem_b0 = [&](int m) { return rec[8 + 4 * m + 1]; };
  auto mem_slot = [&](int m) { return rec[8 + 4 * m + 2]; };
  auto seq_in_range = [&](int m) { return mem_seq(m) >= 0 && mem_seq(m) < a.B; };

  // ------------------------------------------------------------ loads that depend only on the record
  // Issued together, before any is used: the members' first-block words and query
  // positions, the queries, and (below) the team's block words.
  // A member's offset p comes from its own word for the run's first block, whose
  // physical id must be the one the item loads (the source's).
  uint32_t w_mem = 0u, w_src = 0u;
  int qp_mem = 0;
  const float2 t_freq = __ldg(&a.rope[threadIdx.x % HALF]);  // the only frequency this thread evaluates
  bool mem_good = false;
  if (threadIdx.x < nmem) {
    const int m = threadIdx.x, seq = mem_seq(m), bm = mem_b0(m), slot = mem_slot(m);
    mem_good = seq_in_range(m) && bm >= 0 && bm <= a.max_blocks - nblk && slot >= 0 && slot < a.num_slots;
    if (mem_good) {
      w_mem = __ldg(&a.words[(size_t)seq * a.max_blocks + bm]);
      w_src = __ldg(&a.words[(size_t)src * a.max_blocks + b0]);
      qp_mem = __ldg(&a.q_pos[seq]);
    }
  }
  // Each lane's query elements: rows rt*16 + g and + 8, columns 16 ks + 2t + {0, 1, 8, 9}
  // and their rotate-half partners + D/2 (bf16 pairs).
  const int rows = nmem * a.G;
  const int RT = rows <= 16 ? 1 : (rows <= 32 ? 2 : 4);
  const int rt = warp % RT;
  const int g = lane >> 2, t = lane & 3;
  // FP8 (permuted order): dims 32t .. 32t + 31 of each row and their rotate-half
  // partners, as 16-byte vectors.
  constexpr int QV = FP8 ? 4 : 1;
  uint32_t qx[2][NQ][2], qy[2][NQ][2];
  uint4 qo[2][QV], qp[2][QV];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rt * 16 + g + 8 * rr;
    const int m = r / a.G, h = r - m * a.G;
    const bool live = r < rows && seq_in_range(m);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                             ((size_t)(live ? mem_seq(m) : 0) * a.Hq +
                                                              (size_t)kvh * a.G + (live ? h : 0)) * D);
    if constexpr (FP8) {
      const uint4* own = reinterpret_cast<const uint4*>(qrow + 16 * t);        // dims 32t ..
      const uint4* par = reinterpret_cast<const uint4*>(qrow + 16 * (t ^ 2));  // dims (32t) ^ 64 ..
#pragma unroll
      for (int v = 0; v < QV; ++v) {
        qo[rr][v] = live ? __ldg(own + v) : make_uint4(0, 0, 0, 0);
        qp[rr][v] = live ? __ldg(par + v) : make_uint4(0, 0, 0, 0);
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < NQ; ++ks)
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = 16 * ks + 2 * t + 8 * e2;
          qx[rr][ks][e2] = live ? __ldg(qrow + i / 2) : 0u;
          qy[rr][ks][e2] = live ? __ldg(qrow + (i + HALF) / 2) : 0u;
        }
    }
  }

  // ------------------------------------------------------------ teams and first loads
  const int TEAMS = kShWarps / RT;
  const int NS = C::STAGES / TEAMS;  // ring stages of each team: 2, 4 or 8 (twice that for e4m3)
  const int team = warp / RT;
  const int per_team = (nblk + TEAMS - 1) / TEAMS;
  const int kb0 = team * per_team;
  const int nk = max(0, min(nblk, kb0 + per_team) - kb0);  // blocks of this team
  uint8_t* tst = ring + team * NS * C::STAGE_BYTES;
  uint8_t* tconv = ring + C::RING_BYTES + team * G::KV_BYTES;  // FP8: the team's f16 V tile
  auto issue = [&](uint8_t* stage, uint64_t* bar, int phys) {
    if constexpr (FP8) load_block_fp8(stage, bar, phys, a.num_pool_blocks, a.Hkv, kvh, &kmap, &vmap);
    else load_block_3d<D>(stage, bar, phys, a.num_pool_blocks, a.Hkv, kvh, &kmap, &vmap);
  };
  uint64_t* tfull = full + team * NS;
  const bool leader = (rt == 0 && lane == 0);
  const uint32_t* wrow = a.words + (size_t)src * a.max_blocks + b0 + kb0;  // the team's block words
  const uint32_t id_mask = (1u << a.id_bits) - 1u;
  // Physical id the record gives for item block kb < kRecBlocks.
  auto rec_id = [&](int kb) { return rec[kRecIds + kb]; };
  // Lane l describes team block kc + l: physical id (num_pool_blocks = do not load)
  // and valid slots. The block word decides; where the record also names the block,
  // the two must agree, else the block is skipped (its first load may have used the
  // record's id) and the layout error is raised.
  auto describe = [&](int kc, int& phys, int& nv) {
    const int k = kc + lane;
    phys = a.num_pool_blocks;
    nv = 0;
    if (k < nk) {
      const int ph = (int)(__ldg(&wrow[k]) & id_mask);
      if (kb0 + k < kRecBlocks && rec_id(kb0 + k) != ph) {
        raise_status(a.status, LAZY_DEV_LAYOUT);
      } else if (ph < a.num_pool_blocks) {
        phys = ph;
        nv = (kb0 + k == nblk - 1) ? last_nv : kBlock;
      } else {
        raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
      }
    }
  };
  // First loads straight from the record's ids when it names all of them: they need
  // not wait for the block words (which check them below).
  const int pro = min(NS, nk);
  const bool rec_first = kb0 + pro <= kRecBlocks;  // uniform over the team
  if (rec_first && leader)
    for (int k = 0; k < pro; ++k) {
      const int rid = rec_id(kb0 + k);
      const int phys = (rid >= 0 && rid < a.num_pool_blocks) ? rid : a.num_pool_blocks;
      issue(tst + k * C::STAGE_BYTES, &tfull[k], phys);
    }
  int cur_phys, cur_nv, nxt_phys = a.num_pool_blocks, nxt_nv = 0;
  describe(0, cur_phys, cur_nv);
  if (nk > 32) describe(32, nxt_phys, nxt_nv);
  if (!rec_first)
    for (int k = 0; k < pro; ++k) {
      const int phys = __shfl_sync(0xffffffffu, cur_phys, k);
      if (leader) issue(tst + k * C::STAGE_BYTES, &tfull[k], phys);
    }
  int issued = pro;
  LAZY_TRACE(1, global_timer_ns());

  if (threadIdx.x < nmem) {
    const int m = threadIdx.x;
    bool good = mem_good;
    int delta = 0;
    if (good) {
      const BlockInfo mi = decode_word(w_mem, mem_b0(m), a.id_bits);
      good = mi.phys == decode_word(w_src, b0, a.id_bits).phys;
      delta = LAZY ? qp_mem - mi.p : qp_mem;
    }
    if (!good) raise_status(a.status, LAZY_DEV_LAYOUT);
    m_ok[m] = good;
    m_delta[m] = delta;
  }
  __syncthreads();  // m_delta, m_ok

  // ------------------------------------------------------------ rotated query fragments
  // (cos, sin)(delta_m w_f) for every member m and frequency f; each pair is rotated
  // by the lane that holds both halves, scaled by sm_scale * log2(e), rounded to bf16.
  static_assert(kShThreads % HALF == 0, "each thread evaluates one frequency");
  for (int idx = threadIdx.x; idx < nmem * HALF; idx += kShThreads)
    cs_tab[idx] = rope_cs(t_freq, m_delta[idx / HALF], a.status);
  __syncthreads();
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = rt * 16 + g + 8 * rr;
    const int m = r / a.G;
    const float2* cs = cs_tab + (r < rows ? m : 0) * HALF;
    const float sc = (r < rows && m_ok[r < rows ? m : 0]) ? a.scale_log2 : 0.f;  // a failed member's rows are 0
    if constexpr (FP8) {
      // f16 fragments in the permuted order: k-step ks, columns 2t + {0,1} / 2t + 8 + {0,1}
      // hold dims 32t + 4ks + {0,1} / {2,3}; lanes t = 0, 1 hold first halves of
      // rotate-half pairs (x c - y s), t = 2, 3 second halves (y c + x s).
      const bool second = t >= 2;
      const uint32_t* ow = reinterpret_cast<const uint32_t*>(qo[rr]);
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(qp[rr]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        float v[4];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[2 * ks + e2]));
          const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pw[2 * ks + e2]));
          const int f = (32 * t + 4 * ks + 2 * e2) & (HALF - 1);
          const float2 c0 = cs[f], c1 = cs[f + 1];
          const float s0 = second ? c0.y : -c0.y, s1 = second ? c1.y : -c1.y;
          v[2 * e2] = fmaf(x.x, c0.x * sc, y.x * (s0 * sc));
          v[2 * e2 + 1] = fmaf(x.y, c1.x * sc, y.y * (s1 * sc));
        }
        qa[ks][rr] = pack_f16x2(v[0], v[1]);
        qa[ks][rr + 2] = pack_f16x2(v[2], v[3]);
      }
      continue;
    }
#pragma unroll
    for (int ks = 0; ks < NQ; ++ks)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int i = 16 * ks + 2 * t + 8 * e2;
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qx[rr][ks][e2]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qy[rr][ks][e2]));
        float2 c0 = cs[i], c1 = cs[i + 1];
        c0.x *= sc, c0.y *= sc, c1.x *= sc, c1.y *= sc;
        qa[ks][rr + 2 * e2] = pack_bf16x2(fmaf(x.x, c0.x, -y.x * c0.y), fmaf(x.y, c1.x, -y.y * c1.y));
        qa[ks + NQ][rr + 2 * e2] = pack_bf16x2(fmaf(y.x, c0.x, x.x * c0.y), fmaf(y.y, c1.x, x.y * c1.y));
      }
  }
  LAZY_TRACE(2, global_timer_ns());
  // ALiBi (key-position words): a member's word gives the position of its first item
  // block, so delta_r = m - that position and key k of item block kb sits at
  // n - m = 16 kb + k - delta_r; row r's scores get slope_r (n - m) in log2 units.
  float ab_slope[2] = {0.f, 0.f};
  int ab_delta[2] = {0, 0};
  if constexpr (ALIBI) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = rt * 16 + g + 8 * rr;
      const int m = r / a.G, h = r - m * a.G;
      if (r < rows && m_ok[m]) {
        ab_slope[rr] = __ldg(&a.alibi[kvh * a.G + h]) * 1.4426950408889634f;
        ab_delta[rr] = m_delta[m];
      }
    }
  }

  // ------------------------------------------------------------ main loop
  float o[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  const LdsmLane ln = ldsm_lane(lane);
  bool nxt_ready = true;  // nxt holds chunk 32 (or nothing)
  int k = 0;
  for (; k < nk; ++k) {
    if (k > 0 && (k & 31) == 0) {  // advance the word chunk
      cur_phys = nxt_phys;
      cur_nv = nxt_nv;
      nxt_ready = false;
    }
    const int slot = k % NS;
    const int nvalid = __shfl_sync(0xffffffffu, cur_nv, k & 31);
    bool ok = warp_wait(&tfull[slot], (k / NS) & 1, a.status);
    if constexpr (FP8) {
      uint8_t* stage = tst + slot * C::STAGE_BYTES;
      if (ok) convert_fp8_block(stage, tconv, 32 * rt + lane, 32 * RT);
      // the team's f16 V tile is complete before any of its warps reads it
      if (RT > 1) ok = team_and(team, 32 * RT, ok);
      else __syncwarp();
      if (ok)
        attend_block_fp8(smem_u32(stage), smem_u32(tconv), ln, qa, nvalid, o, m_r, l_r, lane, a.k_scale);
    } else if (ok) {
      if constexpr (ALIBI) {
        const int j0 = kBlock * (kb0 + k);
        const float b0[2] = {ab_slope[0] * (float)(j0 - ab_delta[0]), ab_slope[1] * (float)(j0 - ab_delta[1])};
        attend_block_bias<D>(smem_u32(tst + slot * G::STAGE_BYTES), ln, qa, nvalid, o, m_r, l_r, lane, b0, ab_slope);
      } else {
        attend_block<D>(smem_u32(tst + slot * G::STAGE_BYTES), ln, qa, nvalid, o, m_r, l_r, lane);
      }
    }
    // The team's warps are all done with this stage (and agree to go on) before it is refilled.
    if (RT > 1) ok = team_and(team, 32 * RT, ok);
    if (!ok) {
      abort_flag = 1;
      break;
    }
    __syncwarp();
    // Refill this stage with the team's block NS positions ahead.
    const int kn = k + NS;
    if (kn < nk) {
      int phys;
      if ((kn >> 5) == (k >> 5)) {
        phys = __shfl_sync(0xffffffffu, cur_phys, kn & 31);
      } else {
        if (!nxt_ready) {
          describe(kn & ~31, nxt_phys, nxt_nv);
          nxt_ready = true;
        }
        phys = __shfl_sync(0xffffffffu, nxt_phys, kn & 31);
      }
      if (leader) issue(tst + slot * C::STAGE_BYTES, &tfull[slot], phys);
      issued = kn + 1;
    }
  }
  // Copies still in flight (only after a timeout) must land before exit (bounded).
  if (leader)
    for (int kk = k; kk < issued; ++kk) mbar_wait(&tfull[kk % NS], (kk / NS) & 1, a.status);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 1);
    l_r[rr] += __shfl_xor_sync(0xffffffffu, l_r[rr], 2);
  }

  // ------------------------------------------------------------ partials
  // One fp32 partial (m, l, o) per (member, query head) in the member's slot. A
  // member that failed its checks leaves an empty partial (weight 0 in the combine).
  __syncthreads();  // every team is done with its ring (the merge reuses it)
  LAZY_TRACE(3, global_timer_ns());
  if (abort_flag) return;
  float vsc = 1.f;  // FP8: values are code * v_scale, and the output is linear in them
  if constexpr (FP8) vsc = a.v_scale;
  if (TEAMS == 1) {  // one team: write straight from the accumulators
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = rt * 16 + g + 8 * rr;
      if (r >= rows) continue;
      const int m = r / a.G, h = r - m * a.G;
      if (mem_slot(m) < 0 || mem_slot(m) >= a.num_slots) continue;
      const bool good = m_ok[m];
      const size_t pidx = (size_t)mem_slot(m) * a.Hq + (size_t)kvh * a.G + h;
      float* dst = a.ws_o + pidx * D + 2 * t;
#pragma unroll
      for (int j = 0; j < D / 8; ++j)
        *reinterpret_cast<float2*>(dst + 8 * j) =
            good ? make_float2(o[j][2 * rr] * vsc, o[j][2 * rr + 1] * vsc) : make_float2(0.f, 0.f);
      if (t == 0) *reinterpret_cast<float2*>(a.ws_ml + 2 * pidx) = good ? make_float2(m_r[rr], l_r[rr])
                                                                         : make_float2(-INFINITY, 0.f);
    }
  } else {  // teams merge through shared memory, one warp per row, D/32 columns per lane
    float* red = reinterpret_cast<float*>(ring);  // [TEAMS][RT*16][RED_STRIDE]
    const int trows = RT * 16;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = rt * 16 + g + 8 * rr;
      if (row < rows) {
        float* dst = red + ((size_t)team * trows + row) * C::RED_STRIDE;
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          *reinterpret_cast<float2*>(dst + 8 * j + 2 * t) = make_float2(o[j][2 * rr] * vsc, o[j][2 * rr + 1] * vsc);
        if (t == 0) *reinterpret_cast<float2*>(dst + D) = make_float2(m_r[rr], l_r[rr]);
      }
    }
    __syncthreads();
    constexpr int PER = D / 32;
    for (int r = warp; r < rows; r += kShWarps) {
      const int m = r / a.G, h = r - m * a.G;
      if (mem_slot(m) < 0 || mem_slot(m) >= a.num_slots) continue;
      const bool good = m_ok[m];
      float M = -INFINITY;
      if (good)
        for (int tm = 0; tm < TEAMS; ++tm) M = fmaxf(M, red[((size_t)tm * trows + r) * C::RED_STRIDE + D]);
      float acc[PER], L = 0.f;
#pragma unroll
      for (int c = 0; c < PER; ++c) acc[c] = 0.f;
      if (M != -INFINITY) {
        for (int tm = 0; tm < TEAMS; ++tm) {
          const float* srow = red + ((size_t)tm * trows + r) * C::RED_STRIDE;
          const float w = fast_ex2(srow[D] - M);
          L += w * srow[D + 1];
#pragma unroll
          for (int c = 0; c < PER; ++c) acc[c] += w * srow[PER * lane + c];
        }
      }
      const size_t pidx = (size_t)mem_slot(m) * a.Hq + (size_t)kvh * a.G + h;
      float* dst = a.ws_o + pidx * D + PER * lane;
      if constexpr (PER == 4)
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      else
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
      if (lane == 0) *reinterpret_cast<float2*>(a.ws_ml + 2 * pidx) = make_float2(M, L);
    }
  }
#ifdef LAZY_DECODE_TRACE
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    LAZY_TRACE(4, global_timer_ns());
    LAZY_TRACE(5, ((uint64_t)item << 16) | smid);
    LAZY_TRACE(6, ((uint64_t)nblk << 16) | (uint64_t)RT);
  }
#endif
}

// ------------------------------------------------------------------ combine
// out[s][h] = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k over the sequence's
// slots k in [slot_indptr[s], slot_indptr[s+1]); a sequence without slots gets 0.
// One warp per (sequence, query head), D/32 output columns per lane. Slots are
// taken BATCH (12 or 16) at a time with all their loads issued together (one
// memory round trip per batch), folded in with the online rescale of the running
// maximum. Launched as a programmatic dependent of the decode kernel: its CTAs
// may become resident while the decode kernel's last CTAs run, and wait for the
// decode grid's completion (and its partials) before reading anything.
template <int D, int BATCH>
__global__ void shared_combine_kernel(const SharedDecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int wg = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wg >= a.B * a.Hq) return;
  const int s = wg / a.Hq, h = wg - s * a.Hq;
  int k0 = a.slot_indptr[s], k1 = a.slot_indptr[s + 1];
  if (k0 < 0 || k1 < k0 || k1 > a.num_slots) {
    if (lane == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
    k0 = k1 = 0;
  }
  constexpr int PER = D / 32;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml);
  float M = -INFINITY, L = 0.f;
  float acc[PER];
#pragma unroll
  for (int c = 0; c < PER; ++c) acc[c] = 0.f;
  for (int kc = k0; kc < k1; kc += BATCH) {
    const int n = min(BATCH, k1 - kc);
    float2 mlj[BATCH];
    float vj[BATCH][PER];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      mlj[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int c = 0; c < PER; ++c) vj[u][c] = 0.f;
      if (u < n) {
        const size_t pidx = (size_t)(kc + u) * a.Hq + h;
        mlj[u] = ml[pidx];
        const float* src = a.ws_o + pidx * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          vj[u][0] = v.x, vj[u][1] = v.y, vj[u][2] = v.z, vj[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          vj[u][0] = v.x, vj[u][1] = v.y;
        }
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) Mn = fmaxf(Mn, mlj[u].x);
    if (Mn == -INFINITY) continue;  // only empty slots so far
    const float r = fast_ex2(M - Mn);  // 0 while nothing was folded in
    L *= r;
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] *= r;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const float w = fast_ex2(mlj[u].x - Mn);  // an empty slot (m = -inf) weighs 0
      L = fmaf(w, mlj[u].y, L);
#pragma unroll
      for (int c = 0; c < PER; ++c) acc[c] = fmaf(w, vj[u][c], acc[c]);
    }
    M = Mn;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (size_t)wg * D + lane * PER;
  if constexpr (PER == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

// ------------------------------------------------------------------ launchers

template <int D, bool LAZY, bool ALIBI, bool FP8 = false>
static cudaError_t launch_shared_t(const SharedDecodeArgs& a, const float* alibi, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, cudaStream_t st, float k_scale = 1.f,
                                   float v_scale = 1.f) {
  using C = SharedCfg<D, FP8>;
  auto kern = decode_shared_kernel<D, LAZY, ALIBI, FP8>;
  cudaError_t e = set_smem_once<decode_shared_kernel<D, LAZY, ALIBI, FP8>>(C::SMEM);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)a.num_items * a.Hkv;
  if constexpr (ALIBI) {
    SharedAlibiArgs aa;
    static_cast<SharedDecodeArgs&>(aa) = a;
    aa.alibi = alibi;
    kern<<<(unsigned)blocks, kShThreads, C::SMEM, st>>>(aa, kmap, vmap);
  } else if constexpr (FP8) {
    (void)alibi;
    SharedFp8Args fa;
    static_cast<SharedDecodeArgs&>(fa) = a;
    fa.k_scale = k_scale;
    fa.v_scale = v_scale;
    kern<<<(unsigned)blocks, kShThreads, C::SMEM, st>>>(fa, kmap, vmap);
  } else {
    (void)alibi;
    kern<<<(unsigned)blocks, kShThreads, C::SMEM, st>>>(a, kmap, vmap);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_shared(const SharedDecodeArgs& a, const float* alibi, bool lazy, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t st) {
  if (a.num_items == 0) return cudaSuccess;
  if (alibi) {  // ALiBi needs the members' positions: lazy mode only
    if (!lazy) return cudaErrorInvalidValue;
    return a.D == 128 ? launch_shared_t<128, true, true>(a, alibi, kmap, vmap, st)
                      : launch_shared_t<64, true, true>(a, alibi, kmap, vmap, st);
  }
  if (a.D == 128)
    return lazy ? launch_shared_t<128, true, false>(a, nullptr, kmap, vmap, st)
                : launch_shared_t<128, false, false>(a, nullptr, kmap, vmap, st);
  return lazy ? launch_shared_t<64, true, false>(a, nullptr, kmap, vmap, st)
              : launch_shared_t<64, false, false>(a, nullptr, kmap, vmap, st);
}

cudaError_t launch_decode_shared_fp8(const SharedDecodeArgs& a, float k_scale, float v_scale, bool lazy,
                                     const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st) {
  if (a.num_items == 0) return cudaSuccess;
  if (a.D != 128) return cudaErrorNotSupported;
  return lazy ? launch_shared_t<128, true, false, true>(a, nullptr, kmap, vmap, st, k_scale, v_scale)
              : launch_shared_t<128, false, false, true>(a, nullptr, kmap, vmap, st, k_scale, v_scale);
}

cudaError_t launch_shared_combine(const SharedDecodeArgs& a, cudaStream_t st) {
  const int warps = a.B * a.Hq;
  if (warps == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Slots per round trip: 12 when sequences hold at most 12 slots on average (one
  // round trip for most, two CTAs per SM), else 16 (fewer round trips).
  const bool wide = (long long)a.num_slots > 12LL * a.B;
  if (a.D == 128)
    return wide ? cudaLaunchKernelEx(&cfg, shared_combine_kernel<128, 16>, a)
                : cudaLaunchKernelEx(&cfg, shared_combine_kernel<128, 12>, a);
  return wide ? cudaLaunchKernelEx(&cfg, shared_combine_kernel<64, 16>, a)
              : cudaLaunchKernelEx(&cfg, shared_combine_kernel<64, 12>, a);
}

}  // namespace lazy
