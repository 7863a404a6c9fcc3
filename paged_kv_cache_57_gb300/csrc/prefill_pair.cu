// prefill_pair.cu -- LazyAttention prefill with two query tiles per CTA (sm_103a).
//
// The method of prefill.cu ("Resumo Técnico: LazyAttention", "Implementação
// Técnica", item 1: one relative rotation R_p per K block, Q rotated once by R_m),
// organised so that every loaded and rotated K/V tile serves 2 x 128 query rows:
// tile A and tile B are q-heads h and h+1 of the same KV head, the same 128 chunk
// rows. The rotation then costs 3/(4*256) of the tile's tensor work per K tile,
// and the two tiles ping-pong: while the softmax warps of one tile compute
// exponentials, the tensor core runs the other tile's products.
//
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B (thread = query row =
//               TMEM lane). S is read from TMEM in 32-column chunks, twice: once
//               for the row maximum, once for the weights, which are written back
//               as bf16 pairs over the first 64 columns of the tile's own S (P
//               stays in TMEM and is the A operand of P V).
//   warps 8-11  K rotation (R_p per 16-row block, in shared memory) and V holes.
//   warp 12     TMA producer of Q_A, Q_B and the K ring (x2); warp 14 of the V ring
//               (x2). A tile is 16 boxes of 16 rows x 64 columns, issued by 16 lanes
//               at once: small TMA boxes only stream fast when many are in flight.
//   warp 13     TMEM owner (512 columns: S_A/P_A, S_B/P_B, O_A, O_B) and MMA issuer,
//               in the order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1).
// Each tile has its own S/P columns, so the two tiles never wait for each other.
// S_t(j+1) overwrites the P_t(j) that PV_t(j) reads, so the MMA warp issues it only
// after PV_t(j) has completed; the softmax of tile t(j+1) therefore always finds
// PV_t(j) done and may rescale O_t without a further wait.
#include <climits>

#include "prefill_common.cuh"

namespace lazy {

namespace {

using namespace pf;

constexpr int NK = 2, NV = 2;
constexpr int THREADS = 480;  // 15 warps
constexpr int TMEM_COLS = 512;

constexpr int OFF_QA = 0;
constexpr int OFF_QB = OFF_QA + TILE;
constexpr int OFF_K = OFF_QB + TILE;
constexpr int OFF_V = OFF_K + NK * TILE;
constexpr int OFF_KMETA = OFF_V + NV * TILE;
constexpr int OFF_VMETA = OFF_KMETA + NK * BLOCKS * (int)sizeof(KMeta);
constexpr int OFF_BAR = OFF_VMETA + NV * BLOCKS * (int)sizeof(VMeta);
constexpr int NBARS = 2 + 3 * NK + 3 * NV + 7;
constexpr int OFF_QCS = (OFF_BAR + NBARS * 8 + 15) & ~15;  // float2 [64]: the tiles' base angles
constexpr int OFF_ROWS = OFF_QCS + (D / 2) * 8;  // float2 [24][64]: angles of row offsets 16 k and r
constexpr int OFF_TMEM = OFF_ROWS + kAngleRows * (D / 2) * 8;
constexpr int SMEM = 1024 + OFF_TMEM + 16;
static_assert(OFF_QCS % 16 == 0 && OFF_ROWS % 16 == 0, "angle rows are written as 16-byte vectors");
static_assert(SMEM <= 227 * 1024, "prefill (pair) shared memory");

}  // namespace

template <bool LAZY>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_pair_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ[2] = {base + OFF_QA, base + OFF_QB};
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
  uint64_t* s_full = v_empty + NV;   // [2]: tile A, tile B
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* pv_done = p_full + 2;    // [2]
  uint64_t* mma_drain = pv_done + 2;
  float2* base_cs = reinterpret_cast<float2*>(base + OFF_QCS);
  float2* angle_rows = reinterpret_cast<float2*>(base + OFF_ROWS);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + OFF_TMEM);
  __shared__ int abort_flag;

  const int tile = blockIdx.x, s = blockIdx.z;
  const int h_of[2] = {2 * (int)blockIdx.y, 2 * (int)blockIdx.y + 1};
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
  const int kvh = h_of[0] / a.G;
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
    }
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
      mbar_arrive_expect_tx(q_full, 2 * TILE);
      for (int t = 0; t < 2; ++t) {
        tma_load_3d(sQ[t], &qmap, q_full, 0, h_of[t], q0 + row0);
        tma_load_3d(sQ[t] + HALF, &qmap, q_full, 64, h_of[t], q0 + row0);
      }
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
      if (j * BLOCKS >= cbase + 32) {  // warp-uniform: the tile starts in the next chunk
        cbase += 32;
        wcur = wnext;
        wnext = cbase + 32 + lane < nb ? __ldg(&wrow[cbase + 32 + lane]) : 0u;
      }
      // Lanes 0..BLOCKS-1 describe the tile's blocks; lane BLOCKS takes the next
      // block's word so that the tile's last block knows where the following one starts.
      const int b = j * BLOCKS + min(lane, BLOCKS);
      const int rel = b - cbase;  // 0 .. 40
      const uint32_t w0 = __shfl_sync(0xffffffffu, wcur, rel & 31);
      const uint32_t w1 = __shfl_sync(0xffffffffu, wnext, rel & 31);
      const uint32_t w = (lane <= BLOCKS && b < nb) ? (rel < 32 ? w0 : w1) : 0u;
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
          vmeta[st * BLOCKS + lane] = VMeta{nv, b >= b_chunk ? kBlock * (b - b_chunk) : -1};
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
      const uint64_t dQ[2] = {sdesc_sw128(smem_u32(sQ[0]), 16, 1024), sdesc_sw128(smem_u32(sQ[1]), 16, 1024)};
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), HALF, 1024);
      auto issue_s = [&](int j, int t) {
        const uint64_t k0 = dK + (uint64_t)(((j % NK) * TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * HALF + (ks & 3) * 32) >> 4;
          tc_mma(tmem + 128 * t, dQ[t] + off, k0 + off, idS, ks > 0);
        }
        tc_commit(&s_full[t]);
      };
      auto issue_pv = [&](int j, int t) {
        const uint64_t v0 = dV + (uint64_t)(((j % NV) * TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)  // P_t: 8 TMEM columns (16 keys) per k-step
          tc_mma_ta(tmem + 256 + 128 * t, tmem + 128 * t + 8 * ks, v0 + (uint32_t)(ks * 2048 >> 4), idO,
                    (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&pv_done[t]);
      };
      bool ok = mbar_wait(q_ready, 0, a.status) && mbar_wait(&k_ready[0], 0, a.status);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(0, 1);
        tc_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const bool more = j + 1 < n_tiles;
        ok = mbar_wait(&p_full[0], j & 1, a.status) && mbar_wait(&v_full[j % NV], (j / NV) & 1, a.status) &&
             mbar_wait(&v_ready[j % NV], (j / NV) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j, 0);
        if (more) {  // S_A(j+1) overwrites P_A(j): wait for PV_A(j)
          ok = mbar_wait(&k_ready[(j + 1) % NK], ((j + 1) / NK) & 1, a.status) && mbar_wait(&pv_done[0], j & 1, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1, 0);
        }
        ok = mbar_wait(&p_full[1], j & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j, 1);
        tc_commit(&v_empty[j % NV]);
        if (more) {
          ok = mbar_wait(&pv_done[1], j & 1, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1, 1);
          tc_commit(&k_empty[(j + 1) % NK]);
        }
      }
      if (!ok) abort_flag = 1;
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
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
      bool holes = false;
#pragma unroll 1
      for (int bl = 0; bl < BLOCKS; ++bl) {
        const KMeta m = kmeta[st * BLOCKS + bl];
        holes |= m.nvalid < kBlock;
        if constexpr (LAZY) {
          if (m.nvalid > 0) {
            if (m.p != p_cached) {
              float2 cs[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) cs[e] = rope_cs(tr[e], m.p, a.status);
              rot = make_rot8(cs, 1.f);
              p_cached = m.p;
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
      fence_proxy_async_smem();
      mbar_arrive(&k_ready[st]);
      // v_ready(j) is arrived only after V(j) has landed, so no v_ready phase can run
      // two tiles ahead of the MMA warp (V(j+2) needs the P V products of tile j first).
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
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax, tile t
    const int t = warp >> 2;
    const int i = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const int iq = row0 + i;          // query index within the chunk
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + 128 * t, tO = tmem + 256 + 128 * t;
    // Q prologue: q_i' = R_{m_i} q_i, pre-scaled by sm_scale * log2(e); both tiles
    // hold rows at m_i = q_start + row0 + i.
    if (threadIdx.x < D / 2) base_cs[threadIdx.x] = rope_cs(__ldg(&a.rope[threadIdx.x]), a.q_start[s] + row0, a.status);
    load_angle_rows(angle_rows, a.rope, threadIdx.x, 256);
    named_sync(1, 256);
    bool ok = warp_wait(q_full, 0, a.status);
    if (ok) {
      rotate_q_row(sQ[t], i, 0, 8, base_cs, angle_rows, a.scale_log2);
      fence_proxy_async_smem();
    }
    mbar_arrive(q_ready);
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int vs = j % NV;
      ok = warp_wait(&s_full[t], j & 1, a.status) && warp_wait(&v_full[vs], (j / NV) & 1, a.status);
      if (!ok) break;
      tc_fence_after();
      // Per-block key limits for this row (holes; causal inside the chunk).
      int lim[BLOCKS];
      bool full_tile = true;
#pragma unroll
      for (int bl = 0; bl < BLOCKS; ++bl) {
        const VMeta m = vmeta[vs * BLOCKS + bl];
        full_tile &= (m.nvalid == kBlock) & (m.chunk_j0 < 0);
        lim[bl] = m.chunk_j0 >= 0 ? max(0, min(m.nvalid, iq - m.chunk_j0 + 1)) : m.nvalid;
      }
      // Pass 1: row maximum.
      float mx = -INFINITY;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float sv[32];
        tmem_ld32(tS + lane_base + 32 * q, sv);
        tmem_ld_wait(sv);
        if (full_tile) {
          float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            m2[0] = fmax3(m2[0], sv[k], sv[k + 1]);
            m2[1] = fmax3(m2[1], sv[k + 2], sv[k + 3]);
          }
          mx = fmax3(mx, m2[0], m2[1]);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if ((k & 15) < lim[2 * q + (k >> 4)]) mx = fmaxf(mx, sv[k]);
        }
      }
      // Refresh the running maximum only when it grows by more than 2^8 (weights stay <= 256).
      float alpha = 1.f;
      if (mx > m_run + RESCALE_LOG2) {
        alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
        m_run = mx;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // Pass 2: weights -> bf16 P over S's first 64 columns (chunk q's 16 words land on
      // columns already read), row sum in fp32.
      const uint64_t mm = f2(m_use, m_use);
      uint64_t acc = f2(0.f, 0.f);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float sv[32];
        tmem_ld32(tS + lane_base + 32 * q, sv);
        tmem_ld_wait(sv);
        if (!full_tile) {
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if ((k & 15) >= lim[2 * q + (k >> 4)]) sv[k] = -INFINITY;
        }
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 dv = f2_split(f2_sub(f2(sv[2 * k], sv[2 * k + 1]), mm));
          const float e0 = ex2(dv.x), e1 = ex2(dv.y);
          pw[k] = pack_bf16x2(e0, e1);
          acc = f2_add(acc, f2(e0, e1));
        }
        tmem_st16(tS + lane_base + 16 * q, pw);
      }
      const float2 sa = f2_split(acc);
      l_run = l_run * alpha + (sa.x + sa.y);
      // Rescale the running output when this row's maximum was refreshed (warp-uniform);
      // PV_t(j-1) has completed, since S_t(j) was issued after it.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(tO + lane_base + 32 * q, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tO + lane_base + 32 * q, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
    }
    if (!ok && n_tiles > 0) abort_flag = 1;
    // Epilogue: O / l -> bf16.
    if (ok && n_tiles > 0) ok = warp_wait(&pv_done[t], (n_tiles - 1) & 1, a.status);
    if (ok) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(q0 + iq) * a.Hq + h_of[t]) * D;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float o[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + lane_base + 32 * q, o);
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

cudaError_t launch_prefill_pair(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, cudaStream_t st) {
  if (a.D != D || a.G % 2 != 0) return cudaErrorNotSupported;
  if (a.B == 0 || a.max_q_len == 0) return cudaSuccess;
  dim3 grid((a.max_q_len + BM - 1) / BM, a.Hq / 2, a.B);
  auto kern = lazy ? prefill_pair_kernel<true> : prefill_pair_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, SMEM, st>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace lazy
