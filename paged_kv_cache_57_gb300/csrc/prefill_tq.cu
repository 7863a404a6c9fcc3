// prefill_tq.cu -- LazyAttention prefill, one 128-row query tile per CTA, with the
// rotated Q tile held in tensor memory (sm_103a).
//
// The method of prefill.cu ("Resumo Técnico: LazyAttention", "Implementação
// Técnica", item 1: one relative rotation R_p per K block, Q rotated once by R_m).
// Both products read their A operand from TMEM: S = Q' K^T takes Q' (rotated,
// pre-scaled, bf16) from TMEM and K from shared memory; O += P V takes P from
// TMEM and V from shared memory. An MMA with its A operand in shared memory has to
// fetch that operand from shared memory for every 16-wide k-step, which halves its
// rate at N = 128; with A in TMEM only B is fetched.
//
//   warps 0-7   Q prologue (R_m q -> TMEM), softmax, epilogue. Warps w and w + 4
//               share the 32 TMEM lanes (query rows) of quadrant w & 3; warp w < 4
//               takes key columns 0..63 of each tile, warp w + 4 columns 64..127.
//               The two halves of a row exchange only their maxima (shared memory,
//               a 64-thread named barrier); each keeps its own partial row sum.
//   warps 8-11  K rotation (R_p per 16-row block, in shared memory) and V holes.
//   warp 12     TMA producer of Q and the K ring (x3, 32 KiB stages); warp 14 of the
//               V ring (x2). A tile is 16 boxes of 16 rows x 64 columns, issued by 16
//               lanes at once: small TMA boxes only stream fast when many are in flight.
//   warp 13     TMEM owner and MMA issuer.
// TMEM columns: [0,128) S buffer 0, [128,256) S buffer 1, [256,384) O, [384,448) Q',
// [448,512) P (two bf16 per column). S(j) goes to buffer j & 1: the MMA warp issues
// S(j+2) as soon as the softmax has read S(j), right behind P(j) V(j), and the
// softmax of tile j+1 finds S(j+1) ready. The softmax writes P(j) once P(j-1) V(j-1)
// has completed (that wait also makes O safe to rescale).
// Barriers that could be passed twice before their consumer looks (S ready) come one
// per buffer; the epilogue waits on a barrier with a single phase.
#include <climits>
#include <type_traits>

#include "prefill_common.cuh"

namespace lazy {

namespace {

using namespace pf;

constexpr int NK = 3, NV = 2;
constexpr int THREADS = 480;  // 15 warps
constexpr int TMEM_COLS = 512;
constexpr uint32_t COL_O = 256, COL_Q = 384, COL_P = 448;

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;
constexpr int OFF_V = OFF_K + NK * TILE;
constexpr int OFF_KMETA = OFF_V + NV * TILE;
constexpr int OFF_VMETA = OFF_KMETA + NK * BLOCKS * (int)sizeof(KMeta);
constexpr int OFF_BAR = OFF_VMETA + NV * BLOCKS * (int)sizeof(VMeta);
constexpr int NBARS = 2 + 3 * NK + 3 * NV + 2 + 1 + 1 + 1 + 1;
constexpr int OFF_QCS = (OFF_BAR + NBARS * 8 + 15) & ~15;  // float2 [64]: the tile's base angles
constexpr int OFF_ROWS = OFF_QCS + (D / 2) * 8;  // float2 [24][64]: angles of row offsets 16 k and r
constexpr int OFF_TMEM = OFF_ROWS + kAngleRows * (D / 2) * 8;
constexpr int SMEM = 1024 + OFF_TMEM + 16;
static_assert(OFF_QCS % 16 == 0 && OFF_ROWS % 16 == 0, "angle rows are written as 16-byte vectors");
static_assert(SMEM <= 227 * 1024, "prefill (TMEM Q) shared memory");

// Named barriers (0 is __syncthreads): 1 = the 256 softmax threads, 2 + quadrant =
// the 64 threads that share one quadrant of rows.
constexpr int BAR_SOFTMAX = 1, BAR_PAIR0 = 2;

// Chunks c0 .. c0+3 of row i of the staged Q tile rotated by R_{base+i} and
// pre-scaled, stored as packed bf16 pairs to TMEM lane (lane_base + thread) from
// column tq: dims 0..63 in columns [tq, tq + 32), dims 64..127 in [tq + 32, tq + 64)
// (column w = dims 2w, 2w + 1 of its half).
__device__ __forceinline__ void store_rotated_q(const uint8_t* sQ, int i, int c0, const float2* base_cs,
                                                const float2* sm_rows, float scale, uint32_t tq) {
#pragma unroll 1
  for (int c = c0; c < c0 + 4; ++c) {
    uint4 X = *reinterpret_cast<const uint4*>(sQ + sw128(i, c));
    uint4 Y = *reinterpret_cast<const uint4*>(sQ + HALF + sw128(i, c));
    rotate_chunk(X, Y, row_rot8(base_cs, sm_rows, i, c, scale));
    tmem_st4(tq + 4 * c, X);
    tmem_st4(tq + 32 + 4 * c, Y);
  }
}

}  // namespace

template <bool LAZY, bool ALIBI = false>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_tq_kernel(const std::conditional_t<ALIBI, PrefillAlibiArgs, PrefillArgs> a,
                      const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  static_assert(!(ALIBI && LAZY), "the ALiBi prefill does not rotate");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base + OFF_Q;
  uint8_t* sK = base + OFF_K;
  uint8_t* sV = base + OFF_V;
  KMeta* kmeta = reinterpret_cast<KMeta*>(base + OFF_KMETA);
  VMeta* vmeta = reinterpret_cast<VMeta*>(base + OFF_VMETA);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_ready = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_ready = k_full + NK;
  uint64_t* k_empty = k_ready + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_ready = v_full + NV;
  uint64_t* v_empty = v_ready + NV;
  uint64_t* s_full = v_empty + NV;  // [buffer]
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_done = pv_done + 1;   // the last P V has completed (one phase)
  uint64_t* mma_drain = o_done + 1;
  float2* base_cs = reinterpret_cast<float2*>(base + OFF_QCS);
  float2* angle_rows = reinterpret_cast<float2*>(base + OFF_ROWS);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + OFF_TMEM);
  __shared__ int abort_flag;

  const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = a.cu_seqlens_q[s];
  const int C = a.cu_seqlens_q[s + 1] - q0;
  const int row0 = tile * BM;
  if (row0 >= C) return;  // uniform: this tile holds no query row of the chunk
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  int b_chunk = nb - (C + kBlock - 1) / kBlock;  // the chunk's own keys are the last segment
  if (b_chunk < 0) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    b_chunk = 0;
  }
  const int i_last = min(C, row0 + BM) - 1;
  const int last_block = min(nb - 1, b_chunk + i_last / kBlock);
  const int n_tiles = last_block < 0 ? 0 : last_block / BLOCKS + 1;
  const int kvh = h / a.G;
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_ready, 256);
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_ready[i], 128);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_ready[i], 128);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(p_full, 256);
    mbar_init(pv_done, 1);
    mbar_init(o_done, 1);
    mbar_init(mma_drain, 1);
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 12 || warp == 14) {
    // ---------------------------------------------------------------- TMA producers
    const bool is_v = warp == 14;
    if (!is_v && lane == 0) {
      tma_prefetch_map(&qmap);
      tma_prefetch_map(&kmap);
      mbar_arrive_expect_tx(q_full, TILE);
      tma_load_3d(sQ, &qmap, q_full, 0, h, q0 + row0);
      tma_load_3d(sQ + HALF, &qmap, q_full, 64, h, q0 + row0);
    }
    if (is_v && lane == 0) tma_prefetch_map(&vmap);
    // Block words are read 32 at a time, one chunk ahead: lane l holds the word of
    // block cbase + l (wcur) and of block cbase + 32 + l (wnext).
    int cbase = 0;
    uint32_t wcur = lane < nb ? __ldg(&wrow[lane]) : 0u;
    uint32_t wnext = 32 + lane < nb ? __ldg(&wrow[32 + lane]) : 0u;
    const int ns = is_v ? NV : NK;
    uint64_t* ful_ring = is_v ? v_full : k_full;
    uint64_t* emp_ring = is_v ? v_empty : k_empty;
    uint8_t* ring = is_v ? sV : sK;
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      // ALiBi walks the tiles from the last (the keys nearest the queries, with the
      // largest bias) to the first, so that the running maximum is met early and later
      // tiles seldom raise it (each raise rescales the running output).
      const int jt = ALIBI ? n_tiles - 1 - j : j;
      const int b = jt * BLOCKS + min(lane, BLOCKS);
      uint32_t w;
      if constexpr (ALIBI) {
        w = (lane <= BLOCKS && b < nb) ? __ldg(&wrow[b]) : 0u;
      } else {
        if (j * BLOCKS >= cbase + 32) {  // warp-uniform: the tile starts in the next chunk
          cbase += 32;
          wcur = wnext;
          wnext = cbase + 32 + lane < nb ? __ldg(&wrow[cbase + 32 + lane]) : 0u;
        }
        // Lanes 0..BLOCKS-1 describe the tile's blocks; lane BLOCKS takes the next
        // block's word so that the tile's last block knows where the following one starts.
        const int rel = b - cbase;  // 0 .. 40
        const uint32_t w0 = __shfl_sync(0xffffffffu, wcur, rel & 31);
        const uint32_t w1 = __shfl_sync(0xffffffffu, wnext, rel & 31);
        w = (lane <= BLOCKS && b < nb) ? (rel < 32 ? w0 : w1) : 0u;
      }
      const BlockInfo bi = decode_word(w, b, a.id_bits);
      const int p_after = __shfl_down_sync(0xffffffffu, bi.p, 1);
      int y = -kBlock, nv = 0;  // rows of an invalid block start at -16: read as zeros
      if (lane < BLOCKS && b < nb) {
        nv = block_valid(b, nb, seq_len, bi.p, b + 1 < nb ? p_after : bi.p);
        nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
        if (bi.phys < a.num_pool_blocks) {
          y = (bi.phys * a.Hkv + kvh) * kBlock;
        } else {
          if (!is_v) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
          nv = 0;
        }
      }
      const int ybox = __shfl_sync(0xffffffffu, y, (lane >> 1) & 7);  // lane l loads half l & 1 of block l >> 1
      const int st = j % ns;
      if (j >= ns && !warp_wait(&emp_ring[st], ((j / ns) & 1) ^ 1, a.status)) {
        ok = false;
        break;
      }
      if (lane < BLOCKS) {
        if (is_v)
          vmeta[st * BLOCKS + lane] = VMeta{nv, b >= b_chunk ? kBlock * (b - b_chunk) : -1, bi.p, 0};
        else
          kmeta[st * BLOCKS + lane] = KMeta{bi.p, nv};
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&ful_ring[st], TILE);
      __syncwarp();
      if (lane < 2 * BLOCKS)
        tma_load_2d(ring + st * TILE + (lane & 1) * HALF + (lane >> 1) * (kBlock * 128), map, &ful_ring[st],
                    (lane & 1) * 64, ybox);
      issued = j + 1;
    }
    if (!ok) abort_flag = 1;
    if (lane == 0) {  // every copy issued must land before the CTA exits (bounded)
      if (!is_v) mbar_wait(q_full, 0, a.status);
      for (int j = max(0, issued - ns); j < issued; ++j) mbar_wait(&ful_ring[j % ns], (j / ns) & 1, a.status);
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idO = idesc_bf16_f32(BM, D, true);
      // Descriptors are built once; a byte offset moves the 14-bit start-address
      // field by offset >> 4 (shared addresses stay below 2^18, so it never carries).
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), HALF, 1024);
      auto issue_s = [&](int j) {  // S(j) = Q' K(j)^T into buffer j & 1
        const uint64_t k0 = dK + (uint64_t)(((j % NK) * TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)  // Q': 8 TMEM columns (16 dims) per k-step
          tc_mma_ta(tmem + 128 * (j & 1), tmem + COL_Q + 8 * ks, k0 + (uint32_t)(((ks >> 2) * HALF + (ks & 3) * 32) >> 4),
                    idS, ks > 0);
        tc_commit(&s_full[j & 1]);
      };
      auto issue_pv = [&](int j) {  // O += P(j) V(j)
        const uint64_t v0 = dV + (uint64_t)(((j % NV) * TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)  // P: 8 TMEM columns (16 keys) per k-step
          tc_mma_ta(tmem + COL_O, tmem + COL_P + 8 * ks, v0 + (uint32_t)(ks * 2048 >> 4), idO,
                    (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(pv_done);
        if (j == n_tiles - 1) tc_commit(o_done);
      };
      bool ok = mbar_wait(q_ready, 0, a.status);
      if (ok) tc_fence_after();
      for (int j = 0; ok && j < min(2, n_tiles); ++j) {
        ok = mbar_wait(&k_ready[j % NK], (j / NK) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
        tc_commit(&k_empty[j % NK]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        // p_full(j): P(j) is in TMEM and S(j) has been read, so buffer j & 1 is free.
        ok = mbar_wait(p_full, j & 1, a.status) && mbar_wait(&v_full[j % NV], (j / NV) & 1, a.status) &&
             mbar_wait(&v_ready[j % NV], (j / NV) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
        tc_commit(&v_empty[j % NV]);
        if (j + 2 < n_tiles) {
          ok = mbar_wait(&k_ready[(j + 2) % NK], ((j + 2) / NK) & 1, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 2);
          tc_commit(&k_empty[(j + 2) % NK]);
        }
      }
      if (!ok) abort_flag = 1;
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ---------------------------------------------------------------- K rotation, V holes
    const int t = threadIdx.x - 256;
    const int c = t & 7, r = t >> 3;  // 16-byte chunk (8 frequencies) and row within a block
    float2 tr[8];
    Rot8 rot;
    if constexpr (LAZY) {
#pragma unroll
      for (int e = 0; e < 8; ++e) tr[e] = __ldg(&a.rope[8 * c + e]);
    }
    int p_cached = INT_MIN;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % NK;
      if (!warp_wait(&k_full[st], (j / NK) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      uint8_t* kt = sK + st * TILE;
      KMeta m[BLOCKS];
      bool holes = false, one_doc = true;
#pragma unroll
      for (int bl = 0; bl < BLOCKS; ++bl) {
        m[bl] = kmeta[st * BLOCKS + bl];
        holes |= m[bl].nvalid < kBlock;
        one_doc &= m[bl].p == m[0].p;
      }
      if constexpr (LAZY) {
        if (one_doc && !holes) {
          // Common case: the whole tile is one document, one R_p for all 8 blocks.
          if (m[0].p != p_cached) {
            float2 cs[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) cs[e] = rope_cs(tr[e], m[0].p, a.status);
            rot = make_rot8(cs, 1.f);
            p_cached = m[0].p;
          }
#pragma unroll
          for (int bl = 0; bl < BLOCKS; ++bl) {
            const uint32_t off = bl * (kBlock * 128) + sw128(r, c);
            uint4 X = *reinterpret_cast<uint4*>(kt + off);
            uint4 Y = *reinterpret_cast<uint4*>(kt + HALF + off);
            rotate_chunk(X, Y, rot);
            *reinterpret_cast<uint4*>(kt + off) = X;
            *reinterpret_cast<uint4*>(kt + HALF + off) = Y;
          }
        } else {
#pragma unroll 1
          for (int bl = 0; bl < BLOCKS; ++bl) {
            if (m[bl].nvalid > 0) {
              if (m[bl].p != p_cached) {
                float2 cs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) cs[e] = rope_cs(tr[e], m[bl].p, a.status);
                rot = make_rot8(cs, 1.f);
                p_cached = m[bl].p;
              }
              const uint32_t off = bl * (kBlock * 128) + sw128(r, c);
              uint4 X = *reinterpret_cast<uint4*>(kt + off);
              uint4 Y = *reinterpret_cast<uint4*>(kt + HALF + off);
              rotate_chunk(X, Y, rot);
              *reinterpret_cast<uint4*>(kt + off) = X;
              *reinterpret_cast<uint4*>(kt + HALF + off) = Y;
            }
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&k_ready[st]);
      // v_ready(j) is arrived only after V(j) has landed, and V(j + NV) cannot land
      // before P(j) V(j), so no v_ready phase runs a ring ahead of the MMA warp.
      const int vs = j % NV;
      if (!warp_wait(&v_full[vs], (j / NV) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      if (__any_sync(0xffffffffu, holes)) {  // hole slots' V rows may hold anything: zero them
        uint8_t* vt = sV + vs * TILE;
#pragma unroll 1
        for (int bl = 0; bl < BLOCKS; ++bl) {
          if (r >= vmeta[vs * BLOCKS + bl].nvalid) {
            const uint32_t off = bl * (kBlock * 128) + sw128(r, c);
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vt + HALF + off) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&v_ready[vs]);
    }
  } else {
    // ---------------------------------------------------------------- softmax (half rows)
    const int quad = warp & 3, hc = warp >> 2;  // lane quadrant, key-column half
    const int i = threadIdx.x & 127;            // query row within the tile == TMEM lane
    const int iq = row0 + i;                    // query index within the chunk
    const int pair_bar = BAR_PAIR0 + quad;
    // ALiBi: slope of the query head in log2 units and the row's position m_i.
    float slope2 = 0.f;
    int m_row = 0;
    if constexpr (ALIBI) {
      slope2 = __ldg(&a.alibi[h]) * 1.4426950408889634f;
      m_row = a.q_start[s] + iq;
    }
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const uint32_t tO = tmem + COL_O + lane_base + 64 * hc;  // this thread's 64 columns of O
    const uint32_t tP = tmem + COL_P + lane_base + 32 * hc;  // and its 32 columns of P
    // Q prologue: q_i' = R_{m_i} q_i, pre-scaled by sm_scale * log2(e), to TMEM
    // (this thread: dims 32 hc .. 32 hc + 31 of each half); m_i = q_start + row0 + i.
    if (threadIdx.x < D / 2) base_cs[threadIdx.x] = rope_cs(__ldg(&a.rope[threadIdx.x]), a.q_start[s] + row0, a.status);
    load_angle_rows(angle_rows, a.rope, threadIdx.x, 256);
    named_sync(BAR_SOFTMAX, 256);
    bool ok = warp_wait(q_full, 0, a.status);
    if (ok) {
      store_rotated_q(sQ, i, 4 * hc, base_cs, angle_rows, a.scale_log2,
                      tmem + COL_Q + lane_base);
      tmem_st_wait();
      tc_fence_before();
    }
    mbar_arrive(q_ready);
    named_sync(BAR_SOFTMAX, 256);  // the staged Q tile is no longer read: reuse it
    float* red_m = reinterpret_cast<float*>(sQ);  // [2 tiles][2 halves][128 rows]: row maxima
    float* red_l = red_m + 512;                   // [2 halves][128 rows]: row sums
    float m_run = -INFINITY, l_half = 0.f;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1, vs = j % NV;
      const uint32_t tS = tmem + 128 * b + lane_base + 64 * hc;
      // Every exit from this loop is agreed by the pair at its named barrier.
      ok = ok && warp_wait(&s_full[b], (j >> 1) & 1, a.status) && warp_wait(&v_full[vs], (j / NV) & 1, a.status);
      float sv[2][32];
      int lim[4];
      bool full_half = true;
      float mx = -INFINITY;
      if (ok) {
        tc_fence_after();
        tmem_ld32(tS, sv[0]);
        tmem_ld32(tS + 32, sv[1]);
        // Key limits of this half's 4 blocks (holes; causal inside the chunk), read
        // while the loads are in flight.
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const VMeta m = vmeta[vs * BLOCKS + 4 * hc + k];
          full_half &= (m.nvalid == kBlock) & (m.chunk_j0 < 0);
          lim[k] = m.chunk_j0 >= 0 ? max(0, min(m.nvalid, iq - m.chunk_j0 + 1)) : m.nvalid;
        }
        tmem_ld_wait(sv[0], sv[1]);
        if constexpr (ALIBI) {  // + slope (n - m_i), n = the block's first key position + slot
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const float b0 = slope2 * (float)(vmeta[vs * BLOCKS + 4 * hc + k4].pos - m_row);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              float& x = sv[k4 >> 1][16 * (k4 & 1) + k];
              x = fmaf(slope2, (float)k, x + b0);
            }
          }
        }
        if (!full_half) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if ((k & 15) >= lim[k >> 4]) sv[k >> 5][k & 31] = -INFINITY;
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
        mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
        red_m[(2 * b + hc) * 128 + i] = mx;
      }
      ok = named_and(pair_bar, 64, ok);
      if (!ok) break;
      mx = fmaxf(red_m[(2 * b) * 128 + i], red_m[(2 * b + 1) * 128 + i]);
      // Refresh the running maximum only when it grows by more than 2^8 (weights stay
      // <= 256). Both halves of a row see the same maxima, so they agree on m_run.
      float alpha = 1.f;
      if (mx > m_run + RESCALE_LOG2) {
        alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
        m_run = mx;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // Weights -> bf16 P (this half's 32 columns), partial row sum in fp32.
      const uint64_t mm = f2(m_use, m_use);
      uint64_t acc[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
      uint32_t pw[2][16];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 dv = f2_split(f2_sub(f2(sv[q][2 * k], sv[q][2 * k + 1]), mm));
          const float e0 = ex2(dv.x), e1 = ex2(dv.y);
          pw[q][k] = pack_bf16x2(e0, e1);
          acc[k & 1] = f2_add(acc[k & 1], f2(e0, e1));
        }
      const float2 sa = f2_split(f2_add(acc[0], acc[1]));
      l_half = l_half * alpha + (sa.x + sa.y);
      // P(j-1) V(j-1) must be done before P is overwritten or O rescaled. P(j) V(j)
      // cannot start before this P is ready, so pv_done is at phase j-1 or just past it.
      if (j > 0) {
        ok = warp_wait(pv_done, (j - 1) & 1, a.status);
        if (ok) tc_fence_after();
      }
      if (ok) {
        tmem_st16(tP, pw[0]);
        tmem_st16(tP + 16, pw[1]);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // warp-uniform
#pragma unroll 1
          for (int q = 0; q < 2; ++q) {
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
      mbar_arrive(p_full);
    }
    if (!ok && n_tiles > 0) abort_flag = 1;
    // Epilogue: O / l -> bf16; the two halves of a row add their partial sums.
    red_l[hc * 128 + i] = l_half;
    ok = named_and(pair_bar, 64, ok);
    const float l_run = red_l[i] + red_l[128 + i];
    if (ok && n_tiles > 0) ok = warp_wait(o_done, 0, a.status);
    if (ok) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(q0 + iq) * a.Hq + h) * D + 64 * hc;
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        float o[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + 32 * q, o);
          tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0.f;
        }
        if (iq < C) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 v = make_uint4(pack_bf16x2(o[k] * inv, o[k + 1] * inv), pack_bf16x2(o[k + 2] * inv, o[k + 3] * inv),
                                 pack_bf16x2(o[k + 4] * inv, o[k + 5] * inv), pack_bf16x2(o[k + 6] * inv, o[k + 7] * inv));
            *reinterpret_cast<uint4*>(dst + 32 * q + k) = v;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t launch_prefill_tq(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, cudaStream_t st, const float* alibi) {
  if (a.D != D) return cudaErrorNotSupported;
  if (a.B == 0 || a.max_q_len == 0) return cudaSuccess;
  dim3 grid((a.max_q_len + BM - 1) / BM, a.Hq, a.B);
  if (alibi) {
    cudaError_t e = set_smem_once<prefill_tq_kernel<false, true>>(SMEM);
    if (e != cudaSuccess) return e;
    PrefillAlibiArgs aa;
    static_cast<PrefillArgs&>(aa) = a;
    aa.alibi = alibi;
    prefill_tq_kernel<false, true><<<grid, THREADS, SMEM, st>>>(aa, qmap, kmap, vmap);
    return cudaGetLastError();
  }
  auto kern = lazy ? prefill_tq_kernel<true> : prefill_tq_kernel<false>;
  cudaError_t e = lazy ? set_smem_once<prefill_tq_kernel<true>>(SMEM) : set_smem_once<prefill_tq_kernel<false>>(SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, SMEM, st>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace lazy
