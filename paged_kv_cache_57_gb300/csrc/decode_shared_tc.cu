// decode_shared_tc.cu -- LazyAttention decode over shared document runs on the
// 5th-generation tensor cores, for wide query groups (sm_103a).
//
// The work items, slots and partial results of decode_shared.cu ("Resumo Técnico:
// LazyAttention", "Implementação Técnica", item 2: each member's query is rotated
// once by its relative offset R_{m-p}; the stored keys are read as they are),
// computed with tcgen05. When one KV head serves G >= 8 query heads (MQA, wide
// GQA such as Llama-3.1-70B's 64/8), an item's rows (members x G, at most 128)
// fill the M = 128 rows of one tensor-core tile, and a 64-key tile costs 12 MMA instructions issued by one
// thread instead of hundreds of dependent mma.sync per warp.
//
//   warps 0-3  prologue (member checks, R_{m-p} q pre-scaled -> shared memory),
//              softmax (thread = row = TMEM lane, 64 key columns per tile), epilogue.
//   warp 4     TMA producer of the K ring, warp 5 of the V ring (2 stages each): a
//              key tile is 4 blocks (64 keys); each block's K (or V) rows arrive as
//              two 16-row x 64-column boxes, one per lane.
//   warp 6     TMEM owner and MMA issuer.
// TMEM, 256 columns (two CTAs share an SM): [0,64) S buffer 0, [64,128) S buffer
// 1, [128,256) O. S(j) = Q' K(j)^T (8 MMAs, N = 64, both operands in shared memory)
// goes to buffer j & 1, so S(j+1) is computed while the softmax works on S(j); the
// softmax writes P(j) (bf16 pairs) over the first 32 columns of its buffer and
// O += P(j) V(j) (4 MMAs, N = 128) reads it from there. S(j+2) reuses the buffer:
// it is issued right behind P(j) V(j), and MMAs issued by one thread execute in
// issue order, so P(j) is read before it is overwritten. The items are the plan's
// (the planner's automatic chunk gives this kernel about one item per resident CTA,
// since an item's fixed cost -- record, query rotation, partials -- is a few
// microseconds).
// Keys past the item's last valid slot, and the slots of a block whose word
// disagrees with the item record, get weight 0 and their V rows are zeroed (a
// pool slot that holds no key may hold anything, NaN included).
#include <cfloat>
#include <type_traits>

#include "prefill_common.cuh"

namespace lazy {

namespace {

constexpr int kTcD = 128;
constexpr int kTcRows = 128;                  // MMA M: members x query heads
constexpr int kTcKeys = 64;                   // keys per tile (MMA N of S)
constexpr int kTcBlocks = kTcKeys / kBlock;   // 4 blocks per tile
constexpr int kTcHalf = kTcKeys * 128;        // one 64-column half of a 64-row tile: 8 KiB
constexpr int kTcTile = 2 * kTcHalf;          // K or V of one tile: 16 KiB
constexpr int kTcQHalf = kTcRows * 128;       // one 64-column half of the Q tile: 16 KiB
constexpr int kTcNS = 2;                      // stages of each ring
constexpr int kTcThreads = 224;               // 7 warps
constexpr int kTcMembers = kTcRows / 8;       // G >= 8: at most 16 members
constexpr uint32_t kTcCols = 256;
constexpr uint32_t kColS = 0, kColO = 128;    // S buffer b at kColS + 64 b
constexpr int kItemInts = LAZY_PLAN_ITEM_INTS;
constexpr int kRecIds = 8 + 4 * LAZY_PLAN_MAX_MEMBERS;
constexpr int kRecBlocks = LAZY_PLAN_ITEM_BLOCK_IDS;
constexpr int kBarSoftmax = 1;                // named barrier of the 128 softmax threads

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + 2 * kTcQHalf;
constexpr int OFF_V = OFF_K + kTcNS * kTcTile;
constexpr int OFF_BAR = OFF_V + kTcNS * kTcTile;
constexpr int NBARS = 4 * kTcNS + 7;
constexpr int OFF_REC = (OFF_BAR + NBARS * 8 + 15) & ~15;  // written as int4
constexpr int OFF_MEM = OFF_REC + kItemInts * 4;  // int m_delta[16], m_ok[16]
constexpr int OFF_CS = (OFF_MEM + 2 * LAZY_PLAN_MAX_MEMBERS * 4 + 15) & ~15;  // float2 [8][64]
constexpr int OFF_TMEM = OFF_CS + kTcMembers * (kTcD / 2) * 8;
constexpr int SMEM = 1024 + OFF_TMEM + 16;
static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(OFF_Q % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "swizzled tiles are 1024-byte aligned");
static_assert(OFF_BAR % 8 == 0 && OFF_REC % 16 == 0 && OFF_MEM % 16 == 0 && OFF_CS % 16 == 0 && OFF_TMEM % 4 == 0,
              "shared-memory slots are aligned for their widest access");
static_assert(kItemInts % 4 == 0 && kItemInts / 4 <= kTcThreads, "item record layout");

}  // namespace

// Optional per-CTA timestamps (build with -DLAZY_DECODE_TRACE): 16 x u64 per CTA
// after the partials in the workspace: start, Q' stored, first S seen, softmax loop
// done, partials written, (sm id, item), (tiles, members), first S issued; then
// cycle totals over the tiles: softmax waiting for S, softmax computing, softmax
// waiting for P V, softmax storing P, MMA waiting for P, MMA waiting to issue S.
#ifdef LAZY_DECODE_TRACE
#define LAZY_TC_TRACE(i, v)                                                                                    \
  do {                                                                                                         \
    reinterpret_cast<uint64_t*>(a.ws_ml + 2 * (size_t)a.num_slots * a.Hq)[16 * (size_t)blockIdx.x + (i)] = (v); \
  } while (0)
#define LAZY_TC_CLK(var) const long long var = clock64()
#define LAZY_TC_ACC(acc, a0, a1) acc += (a1) - (a0)
#else
#define LAZY_TC_TRACE(i, v) \
  do {                      \
  } while (0)
#define LAZY_TC_CLK(var)
#define LAZY_TC_ACC(acc, a0, a1)
#endif

template <bool LAZY, bool ALIBI>
__global__ void __launch_bounds__(kTcThreads, 2)
    decode_shared_tc_kernel(const std::conditional_t<ALIBI, SharedAlibiArgs, SharedDecodeArgs> a,
                            const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = pf::align1024(smem_raw);
  uint8_t* sQ = base + OFF_Q;
  uint8_t* sK = base + OFF_K;
  uint8_t* sV = base + OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* k_full = bars;              // [stage] K(j) has landed
  uint64_t* k_empty = k_full + kTcNS;   // [stage] S(j) has completed
  uint64_t* v_full = k_empty + kTcNS;   // [stage] V(j) has landed
  uint64_t* v_empty = v_full + kTcNS;   // [stage] P(j) V(j) has completed
  uint64_t* q_ready = v_empty + kTcNS;
  uint64_t* s_full = q_ready + 1;       // [buffer]
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_done = pv_done + 1;       // the last P V has completed (one phase)
  uint64_t* mma_drain = o_done + 1;
  int* rec = reinterpret_cast<int*>(base + OFF_REC);
  int* m_delta = reinterpret_cast<int*>(base + OFF_MEM);
  int* m_ok = m_delta + LAZY_PLAN_MAX_MEMBERS;
  float2* cs_tab = reinterpret_cast<float2*>(base + OFF_CS);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + OFF_TMEM);

  // The combine kernel may be scheduled once every CTA of this grid has started;
  // it waits for this grid's completion before it reads the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int kvh = blockIdx.x % a.Hkv;
  const int item = blockIdx.x / a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) LAZY_TC_TRACE(0, global_timer_ns());
  if (threadIdx.x < kItemInts / 4)
    reinterpret_cast<int4*>(rec)[threadIdx.x] =
        __ldg(reinterpret_cast<const int4*>(a.items) + (size_t)item * (kItemInts / 4) + threadIdx.x);
  __syncthreads();
  const int src = rec[0], b0 = rec[1], nblk = rec[2], last_nv = rec[3], nmem = rec[4];
  const bool item_ok = src >= 0 && src < a.B && b0 >= 0 && nblk >= 1 && nblk <= a.max_blocks - b0 &&
                       last_nv >= 1 && last_nv <= kBlock && nmem >= 1 && nmem <= kTcMembers &&
                       nmem * a.G <= kTcRows;
  if (!item_ok) {  // uniform over the CTA: nothing is loaded or written
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcNS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(q_ready, 128);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(o_done, 1);
    mbar_init(mma_drain, 1);
    fence_barrier_init();
  }
  if (warp == 6) {
    tmem_alloc(tmem_holder, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int n_tiles = (nblk + kTcBlocks - 1) / kTcBlocks;
  const int rows = nmem * a.G;
  const uint32_t* wrow = a.words + (size_t)src * a.max_blocks + b0;  // the item's block words
  const uint32_t id_mask = (1u << a.id_bits) - 1u;

  if (warp == 4 || warp == 5) {
    // ---------------------------------------------------------------- TMA producers
    // Lane l < 8 loads column half l & 1 of block l >> 1 of the tile. Ids come from
    // the item record (the first 32 blocks) or the block words; an id outside the
    // pool, or a block past the item, is read at row -16, i.e. as zeros.
    const bool is_v = warp == 5;
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    uint64_t* ful = is_v ? v_full : k_full;
    uint64_t* emp = is_v ? v_empty : k_empty;
    uint8_t* ring = is_v ? sV : sK;
    if (lane == 0) tma_prefetch_map(map);
    const int bl = lane >> 1, half = lane & 1;
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % kTcNS;
      int y = -kBlock;
      if (lane < 2 * kTcBlocks) {
        const int b = j * kTcBlocks + bl;
        if (b < nblk) {
          const int phys = b < kRecBlocks ? rec[kRecIds + b] : (int)(__ldg(&wrow[b]) & id_mask);
          if (phys >= 0 && phys < a.num_pool_blocks) y = (phys * a.Hkv + kvh) * kBlock;
        }
      }
      if (j >= kTcNS && !pf::warp_wait(&emp[st], ((j / kTcNS) & 1) ^ 1, a.status)) break;
      if (lane == 0) mbar_arrive_expect_tx(&ful[st], kTcTile);
      __syncwarp();
      if (lane < 2 * kTcBlocks)
        tma_load_2d(ring + st * kTcTile + half * kTcHalf + bl * (kBlock * 128), map, &ful[st], half * 64, y);
      issued = j + 1;
    }
    if (lane == 0)  // every copy issued must land before the CTA exits (bounded)
      for (int j = max(0, issued - kTcNS); j < issued; ++j) mbar_wait(&ful[j % kTcNS], (j / kTcNS) & 1, a.status);
  } else if (warp == 6) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kTcRows, kTcKeys, false);
      constexpr uint32_t idO = idesc_bf16_f32(kTcRows, kTcD, true);
      // Descriptors are built once; a byte offset moves the 14-bit start-address
      // field by offset >> 4 (shared addresses stay below 2^18, so it never carries).
      const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), kTcHalf, 1024);
      auto issue_s = [&](int j) {  // S(j) = Q' K(j)^T into buffer j & 1
        const uint64_t k0 = dK + (uint64_t)(((j % kTcNS) * kTcTile) >> 4);
#pragma unroll
        for (int ks = 0; ks < kTcD / 16; ++ks)
          tc_mma(tmem + kColS + 64 * (j & 1), dQ + (uint64_t)(((ks >> 2) * kTcQHalf + (ks & 3) * 32) >> 4),
                 k0 + (uint64_t)(((ks >> 2) * kTcHalf + (ks & 3) * 32) >> 4), idS, ks > 0 ? 1u : 0u);
        tc_commit(&k_empty[j % kTcNS]);
        tc_commit(&s_full[j & 1]);
      };
      bool ok = mbar_wait(q_ready, 0, a.status);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < min(2, n_tiles); ++j) {
        ok = mbar_wait(&k_full[j % kTcNS], (j / kTcNS) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        if (j == 0) LAZY_TC_TRACE(7, global_timer_ns());
        issue_s(j);
      }
      long long c_wp = 0, c_ws = 0;
      (void)c_wp;
      (void)c_ws;
      for (int j = 0; ok && j < n_tiles; ++j) {
        // p_full(j): P(j) is in TMEM over buffer j & 1 (S(j) has been read).
        LAZY_TC_CLK(m0);
        ok = mbar_wait(p_full, j & 1, a.status) && mbar_wait(&v_full[j % kTcNS], (j / kTcNS) & 1, a.status);
        LAZY_TC_CLK(m1);
        LAZY_TC_ACC(c_wp, m0, m1);
        if (!ok) break;
        tc_fence_after();
        const uint64_t v0 = dV + (uint64_t)(((j % kTcNS) * kTcTile) >> 4);
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks)  // P: 8 TMEM columns (16 keys) per k-step
          tc_mma_ta(tmem + kColO, tmem + kColS + 64 * (j & 1) + 8 * ks, v0 + (uint64_t)((ks * 16 * 128) >> 4), idO,
                    (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&v_empty[j % kTcNS]);
        tc_commit(pv_done);
        if (j == n_tiles - 1) tc_commit(o_done);
        if (j + 2 < n_tiles) {
          // S(j+2) overwrites P(j) in buffer j & 1. MMAs issued by one thread run in
          // issue order, so P(j) V(j), issued above, reads P(j) before S(j+2) writes.
          LAZY_TC_CLK(m2);
          ok = mbar_wait(&k_full[(j + 2) % kTcNS], ((j + 2) / kTcNS) & 1, a.status);
          LAZY_TC_CLK(m3);
          LAZY_TC_ACC(c_ws, m2, m3);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 2);
        }
      }
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
      LAZY_TC_TRACE(12, c_wp);
      LAZY_TC_TRACE(13, c_ws);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- rows: prologue, softmax, epilogue
    const int i = threadIdx.x;  // row of the tile == TMEM lane (warps 0-3, one quadrant each)
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    // Loads that depend only on the record, issued together before any is used: the
    // row's query (row i = member m, query head hh of this KV head), the members'
    // first-block words and query positions, and the first tile's block words.
    const int m = i / a.G, hh = i - m * a.G;
    const int mseq = i < rows ? rec[8 + 4 * m] : -1;
    const bool row_in = mseq >= 0 && mseq < a.B;
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                       ((size_t)(row_in ? mseq : 0) * a.Hq + (size_t)kvh * a.G +
                                                        (row_in ? hh : 0)) * kTcD);
    uint4 X[8], Y[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      X[c] = row_in ? __ldg(qrow + c) : make_uint4(0, 0, 0, 0);
      Y[c] = row_in ? __ldg(qrow + 8 + c) : make_uint4(0, 0, 0, 0);
    }
    uint32_t w_cur = lane < kTcBlocks && lane < nblk ? __ldg(&wrow[lane]) : 0u;
    // Members: the word of a member's first block must name the item's first
    // physical block; its document offset p gives the rotation R_{m-p} (m: the
    // member's query position). The control path (stored keys already rotated)
    // rotates q by R_m.
    if (i < nmem) {
      const int seq = rec[8 + 4 * i], bm = rec[8 + 4 * i + 1], slot = rec[8 + 4 * i + 2];
      bool good = seq >= 0 && seq < a.B && bm >= 0 && bm <= a.max_blocks - nblk && slot >= 0 && slot < a.num_slots;
      uint32_t w_mem = 0u, w_src = 0u;
      int qp = 0;
      if (good) {
        w_mem = __ldg(&a.words[(size_t)seq * a.max_blocks + bm]);
        w_src = __ldg(&wrow[0]);
        qp = __ldg(&a.q_pos[seq]);
      }
      int delta = 0;
      if (good) {
        const BlockInfo mi = decode_word(w_mem, bm, a.id_bits);
        good = mi.phys == decode_word(w_src, b0, a.id_bits).phys;
        delta = LAZY ? qp - mi.p : qp;
      }
      if (!good) raise_status(a.status, LAZY_DEV_LAYOUT);
      m_ok[i] = good;
      m_delta[i] = delta;
    }
    pf::named_sync(kBarSoftmax, 128);
    for (int idx = i; idx < nmem * (kTcD / 2); idx += 128)
      cs_tab[idx] = rope_cs(__ldg(&a.rope[idx & (kTcD / 2 - 1)]), m_delta[idx / (kTcD / 2)], a.status);
    pf::named_sync(kBarSoftmax, 128);
    // q' = R_{delta} q * sm_scale * log2(e), bf16, row i of the 128-byte-swizzled Q
    // tile (dims 0..63 in the first half, 64..127 in the second). Rows past the
    // item's and a failed member's rows are 0.
    {
      const bool live = row_in && m_ok[m];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (live) {
          float2 cs[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) cs[e] = cs_tab[m * (kTcD / 2) + 8 * c + e];
          pf::rotate_chunk(X[c], Y[c], pf::make_rot8(cs, a.scale_log2));
        } else {
          X[c] = Y[c] = make_uint4(0, 0, 0, 0);
        }
        *reinterpret_cast<uint4*>(sQ + sw128(i, c)) = X[c];
        *reinterpret_cast<uint4*>(sQ + kTcQHalf + sw128(i, c)) = Y[c];
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(q_ready);
    if (i == 0) LAZY_TC_TRACE(1, global_timer_ns());

    const uint32_t tO = tmem + kColO + lane_base;
    // ALiBi (key-position words): the member's word gives the position of its first
    // item block, delta = m - that position, and column c of tile jt sits at
    // n - m = 16 (4 jt) + c - delta; the row's scores get slope (n - m) in log2 units.
    float ab_slope = 0.f;
    int ab_delta = 0;
    if constexpr (ALIBI) {
      if (row_in && m_ok[m]) {
        ab_slope = __ldg(&a.alibi[kvh * a.G + hh]) * 1.4426950408889634f;
        ab_delta = m_delta[m];
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    long long c_s = 0, c_c = 0, c_pv = 0, c_st = 0;
    (void)c_s;
    (void)c_c;
    (void)c_pv;
    (void)c_st;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1, st = j % kTcNS;
      LAZY_TC_CLK(s0);
      const uint32_t tS = tmem + kColS + 64 * b + lane_base;
      // Valid slots of the tile's 4 blocks: lane k < 4 checks block 4j + k's word
      // against the record. The words of the next tile are loaded one tile ahead.
      const int bn = (j + 1) * kTcBlocks + lane;
      const uint32_t w_nxt = lane < kTcBlocks && bn < nblk ? __ldg(&wrow[bn]) : 0u;
      int nv = 0;
      if (lane < kTcBlocks) {
        const int blk = j * kTcBlocks + lane;
        if (blk < nblk) {
          const int ph = (int)(w_cur & id_mask);
          if (blk < kRecBlocks && rec[kRecIds + blk] != ph) {
            if (warp == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
          } else if (ph >= a.num_pool_blocks) {
            if (warp == 0) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
          } else {
            nv = blk == nblk - 1 ? last_nv : kBlock;
          }
        }
      }
      int nvb[kTcBlocks];
      bool full_tile = true, zero_v = false;
#pragma unroll
      for (int k = 0; k < kTcBlocks; ++k) {
        nvb[k] = __shfl_sync(0xffffffffu, nv, k);
        full_tile &= nvb[k] == kBlock;
        zero_v |= (j * kTcBlocks + k < nblk) && nvb[k] < kBlock;  // slots a loaded box may fill with anything
      }
      ok = ok && pf::warp_wait(&s_full[b], (j >> 1) & 1, a.status);
      if (j == 0 && i == 0) LAZY_TC_TRACE(2, global_timer_ns());
      LAZY_TC_CLK(s1);
      LAZY_TC_ACC(c_s, s0, s1);
      if (ok) {
        tc_fence_after();
        float sv[2][32];
        tmem_ld32(tS, sv[0]);
        tmem_ld32(tS + 32, sv[1]);
        tmem_ld_wait(sv[0], sv[1]);
        if constexpr (ALIBI) {
          const float base = ab_slope * (float)(kBlock * kTcBlocks * j - ab_delta);
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c) sv[c >> 5][c & 31] += fmaf(ab_slope, (float)c, base);
        }
        if (!full_tile) {
#pragma unroll
          for (int c = 0; c < kTcKeys; ++c)
            if ((c & 15) >= nvb[c >> 4]) sv[c >> 5][c & 31] = -INFINITY;
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            m4[0] = fmax3(m4[0], sv[q][k], sv[q][k + 1]);
            m4[1] = fmax3(m4[1], sv[q][k + 2], sv[q][k + 3]);
            m4[2] = fmax3(m4[2], sv[q][k + 4], sv[q][k + 5]);
            m4[3] = fmax3(m4[3], sv[q][k + 6], sv[q][k + 7]);
          }
        const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        // Refresh the running maximum only when it grows by more than 2^8 (weights
        // stay <= 256); o and l are kept relative to m_run, which the partial records.
        float alpha = 1.f;
        if (mx > m_run + pf::RESCALE_LOG2) {
          alpha = m_run == -INFINITY ? 0.f : pf::ex2(m_run - mx);
          m_run = mx;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        const uint64_t mm = f2(m_use, m_use);
        uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
        uint32_t pw[2][16];
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 dv = f2_split(f2_sub(f2(sv[q][2 * k], sv[q][2 * k + 1]), mm));
            const float e0 = pf::ex2(dv.x), e1 = pf::ex2(dv.y);
            pw[q][k] = pack_bf16x2(e0, e1);
            acc[k & 1] = f2_add(acc[k & 1], f2(e0, e1));
          }
        const float2 sa = f2_split(f2_add(acc[0], acc[1]));
        l_run = l_run * alpha + (sa.x + sa.y);
        if (zero_v) {  // uniform over the CTA
          ok = pf::warp_wait(&v_full[st], (j / kTcNS) & 1, a.status);
          if (ok) {
            const int r = i >> 3, c = i & 7;  // 16 rows x 8 16-byte chunks of a block
            uint8_t* vt = sV + st * kTcTile;
#pragma unroll
            for (int k = 0; k < kTcBlocks; ++k) {
              if (j * kTcBlocks + k < nblk && r >= nvb[k]) {
                const uint32_t off = k * (kBlock * 128) + sw128(r, c);
                *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(vt + kTcHalf + off) = make_uint4(0, 0, 0, 0);
              }
            }
            fence_proxy_async_smem();
          }
        }
        // P(j-1) V(j-1) must be done before O is rescaled (it also keeps this loop
        // from running two phases ahead of the MMA warp on p_full).
        LAZY_TC_CLK(s2);
        LAZY_TC_ACC(c_c, s1, s2);
        if (ok && j > 0) {
          ok = pf::warp_wait(pv_done, (j - 1) & 1, a.status);
          if (ok) tc_fence_after();
        }
        LAZY_TC_CLK(s3);
        LAZY_TC_ACC(c_pv, s2, s3);
        if (ok) {
          tmem_st16(tS, pw[0]);
          tmem_st16(tS + 16, pw[1]);
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // warp-uniform
#pragma unroll 1
            for (int q = 0; q < kTcD / 32; ++q) {
              float o[32];
              tmem_ld32(tO + 32 * q, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] *= alpha;
              tmem_st32(tO + 32 * q, o);
            }
          }
          tmem_st_wait();
          tc_fence_before();
        }
      }
      mbar_arrive(p_full);
      ok = pf::named_and(kBarSoftmax, 128, ok);  // the four warps leave the loop together
      LAZY_TC_CLK(s4);
      LAZY_TC_ACC(c_st, s0, s4);
      if (!ok) break;
      w_cur = w_nxt;
    }
    if (i == 0) {
      LAZY_TC_TRACE(3, global_timer_ns());
      LAZY_TC_TRACE(8, c_s);
      LAZY_TC_TRACE(9, c_c);
      LAZY_TC_TRACE(10, c_pv);
      LAZY_TC_TRACE(11, c_st);
    }
    // ---------------------------------------------------------------- partials
    // One fp32 partial (m, l, o) per (member, query head) in the member's slot, as
    // decode_shared.cu writes it. A failed member leaves an empty partial (weight 0
    // in the combine).
    if (ok) ok = pf::warp_wait(o_done, 0, a.status);
    if (ok) {
      tc_fence_after();
      const int slot = i < rows ? rec[8 + 4 * m + 2] : -1;
      const bool write = i < rows && slot >= 0 && slot < a.num_slots;
      const bool good = write && m_ok[m];
      const size_t pidx = write ? (size_t)slot * a.Hq + (size_t)kvh * a.G + hh : 0;
      float* dst = a.ws_o + pidx * kTcD;
#pragma unroll 1
      for (int q = 0; q < kTcD / 32; ++q) {
        float o[32];
        tmem_ld32(tO + 32 * q, o);
        tmem_ld_wait(o);
        if (write) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + 32 * q + k) =
                good ? make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (write)
        *reinterpret_cast<float2*>(a.ws_ml + 2 * pidx) =
            good ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.f);
    }
#ifdef LAZY_DECODE_TRACE
    if (i == 0) {
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      LAZY_TC_TRACE(4, global_timer_ns());
      LAZY_TC_TRACE(5, ((uint64_t)smid << 32) | (uint32_t)item);
      LAZY_TC_TRACE(6, ((uint64_t)nmem << 16) | (uint32_t)n_tiles);
    }
#endif
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
}

cudaError_t launch_decode_shared_tc(const SharedDecodeArgs& a, const float* alibi, bool lazy,
                                    const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st) {
  if (a.D != kTcD) return cudaErrorNotSupported;
  if (a.num_items == 0) return cudaSuccess;
  const long long blocks = (long long)a.num_items * a.Hkv;
  if (alibi) {
    if (!lazy) return cudaErrorInvalidValue;  // ALiBi needs the members' positions
    cudaError_t e = set_smem_once<decode_shared_tc_kernel<true, true>>(SMEM);
    if (e != cudaSuccess) return e;
    SharedAlibiArgs aa;
    static_cast<SharedDecodeArgs&>(aa) = a;
    aa.alibi = alibi;
    decode_shared_tc_kernel<true, true><<<(unsigned)blocks, kTcThreads, SMEM, st>>>(aa, kmap, vmap);
    return cudaGetLastError();
  }
  cudaError_t e = lazy ? set_smem_once<decode_shared_tc_kernel<true, false>>(SMEM)
                       : set_smem_once<decode_shared_tc_kernel<false, false>>(SMEM);
  if (e != cudaSuccess) return e;
  auto kern = lazy ? decode_shared_tc_kernel<true, false> : decode_shared_tc_kernel<false, false>;
  kern<<<(unsigned)blocks, kTcThreads, SMEM, st>>>(a, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace lazy
