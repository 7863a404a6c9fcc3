// prefill.cu -- LazyAttention prefill on the 5th-generation tensor cores (sm_103a).
//
// Technical summary "Resumo Técnico: LazyAttention", "Implementação Técnica",
// item 1 (Prefilling, compute-bound): K blocks are loaded from the
// position-agnostic cache and each receives ONE relative rotation (by R_p of its
// document, since stored K already carries its local position) instead of an
// unrotate-then-rerotate pass; the query tile is rotated once by R_m. The extra
// work is 3*N*d FLOPs per N-key tile against 4*M*N*d for the tile's two
// matrix products, i.e. 3/(4M): 0.59% at M = 128.
//
// One CTA = one 128-row query tile of one q-head of one chunk. Warp roles:
//   warps 0-3  softmax: rotate the Q tile once (thread = row), then per key tile
//              read S from TMEM, mask (holes; causal inside the chunk), online
//              (max, sum) softmax ("Flash Attention -- tiling") with the running
//              maximum refreshed only when it grows by more than 2^8, write P
//              (bf16, 128-byte swizzled K-major) to shared memory, rescale O in
//              TMEM when needed; finally O / l -> bf16 -> global.
//   warps 4-7  rotation: rotate each 16-row K block of a landed tile in shared
//              memory by R_p (fp32 math, bf16 result); zero V rows of hole slots.
//   warp 8     TMA producer: Q tile; K tiles into a 3-stage ring and V tiles into
//              a 2-stage ring (8 blocks x 2 boxes of 16 rows x 64 columns each).
//   warp 9     TMEM owner and MMA issuer: S = Q K^T (M=N=128, K=d) into TMEM
//              columns [0,128), O += P V into columns [128,256). It issues each
//              product as soon as its inputs are ready, so the S of the next tile
//              overlaps the softmax of the current one, and frees K stages right
//              after their S and V stages right after their P V.
#include <climits>

#include "kernels.h"
#include "tcgen05.cuh"

namespace lazy {

namespace {

constexpr int PF_BM = 128;                 // query rows per tile (MMA M)
constexpr int PF_BN = 128;                 // keys per tile (MMA N of S)
constexpr int PF_D = 128;                  // head dim
constexpr int PF_NK = 3;                   // K stages
constexpr int PF_NV = 2;                   // V stages
constexpr int PF_BLOCKS = PF_BN / kBlock;  // 8 blocks per key tile
constexpr int PF_HALF = PF_BM * 128;       // one 64-column half of a 128-row tile (bytes)
constexpr int PF_TILE = 2 * PF_HALF;       // 32 KiB
constexpr int PF_THREADS = 320;
constexpr int PF_TMEM_COLS = 256;
constexpr float PF_RESCALE_LOG2 = 8.f;     // refresh the running max when it grows by more than this

struct PfKMeta {
  int p;       // document start position
  int nvalid;  // valid slots (0 for blocks past the sequence or with a bad id)
};
struct PfVMeta {
  int nvalid;
  int chunk_j0;  // chunk-local index of the block's first key, or -1 for cached documents
};

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + PF_TILE;
constexpr int OFF_V = OFF_K + PF_NK * PF_TILE;
constexpr int OFF_P = OFF_V + PF_NV * PF_TILE;
constexpr int OFF_KMETA = OFF_P + PF_TILE;
constexpr int OFF_VMETA = OFF_KMETA + PF_NK * PF_BLOCKS * (int)sizeof(PfKMeta);
constexpr int OFF_BAR = OFF_VMETA + PF_NV * PF_BLOCKS * (int)sizeof(PfVMeta);
constexpr int NBARS = 2 + 3 * PF_NK + 3 * PF_NV + 5;
constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
constexpr int PF_SMEM = 1024 + OFF_TMEM + 16;
static_assert(PF_SMEM <= 227 * 1024, "prefill shared memory");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool warp_wait_pf(uint64_t* bar, uint32_t parity, unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
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

}  // namespace

template <bool LAZY>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1024(smem_raw);
  uint8_t* sQ = base + OFF_Q;
  uint8_t* sK = base + OFF_K;
  uint8_t* sV = base + OFF_V;
  uint8_t* sP = base + OFF_P;
  PfKMeta* kmeta = reinterpret_cast<PfKMeta*>(base + OFF_KMETA);
  PfVMeta* vmeta = reinterpret_cast<PfVMeta*>(base + OFF_VMETA);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_ready = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_ready = k_full + PF_NK;
  uint64_t* k_empty = k_ready + PF_NK;
  uint64_t* v_full = k_empty + PF_NK;
  uint64_t* v_ready = v_full + PF_NV;
  uint64_t* v_empty = v_ready + PF_NV;
  uint64_t* s_full = v_empty + PF_NV;
  uint64_t* s_free = s_full + 1;
  uint64_t* p_full = s_free + 1;
  uint64_t* pv_done = p_full + 1;
  uint64_t* mma_drain = pv_done + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + OFF_TMEM);
  __shared__ int abort_flag;

  const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = a.cu_seqlens_q[s];
  const int C = a.cu_seqlens_q[s + 1] - q0;
  const int row0 = tile * PF_BM;
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
  const int i_last = min(C, row0 + PF_BM) - 1;
  const int last_block = min(nb - 1, b_chunk + i_last / kBlock);
  const int n_tiles = last_block < 0 ? 0 : last_block / PF_BLOCKS + 1;
  const int kvh = h / a.G;
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_ready, 128);
    for (int i = 0; i < PF_NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_ready[i], 128);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < PF_NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_ready[i], 128);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 128);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_holder, PF_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_map(&qmap);
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      mbar_arrive_expect_tx(q_full, PF_TILE);
      tma_load_3d(sQ, &qmap, q_full, 0, h, q0 + row0);
      tma_load_3d(sQ + PF_HALF, &qmap, q_full, 64, h, q0 + row0);
    }
    // Lane l < 8 describes block l of a tile; lane 8 reads the block after (hole rule).
    struct Lane {
      int p, nv, y, j0;
    };
    auto describe = [&](int j) {
      const int b = j * PF_BLOCKS + min(lane, PF_BLOCKS);
      const uint32_t w = (lane <= PF_BLOCKS && b < nb) ? __ldg(&wrow[b]) : 0u;
      const BlockInfo bi = decode_word(w, b, a.id_bits);
      const int p_after = __shfl_down_sync(0xffffffffu, bi.p, 1);
      Lane r{bi.p, 0, -kBlock, -1};  // rows of an invalid block start at -16: read as zeros
      if (lane < PF_BLOCKS && b < nb) {
        int nv = block_valid(b, nb, seq_len, bi.p, b + 1 < nb ? p_after : bi.p);
        nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
        if (bi.phys < a.num_pool_blocks) {
          r.y = (bi.phys * a.Hkv + kvh) * kBlock;
        } else {
          raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
          nv = 0;
        }
        r.nv = nv;
        r.j0 = b >= b_chunk ? kBlock * (b - b_chunk) : -1;
      }
      return r;
    };
    auto issue_k = [&](int j, const Lane& d) -> bool {
      const int st = j % PF_NK;
      if (j >= PF_NK && !warp_wait_pf(&k_empty[st], ((j / PF_NK) & 1) ^ 1, a.status)) return false;
      if (lane < PF_BLOCKS) kmeta[st * PF_BLOCKS + lane] = PfKMeta{d.p, d.nv};
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], PF_TILE);
      __syncwarp();
      if (lane < PF_BLOCKS) {
        uint8_t* kd = sK + st * PF_TILE + lane * (kBlock * 128);
        tma_load_2d(kd, &kmap, &k_full[st], 0, d.y);
        tma_load_2d(kd + PF_HALF, &kmap, &k_full[st], 64, d.y);
      }
      return true;
    };
    auto issue_v = [&](int j, const Lane& d) -> bool {
      const int st = j % PF_NV;
      if (j >= PF_NV && !warp_wait_pf(&v_empty[st], ((j / PF_NV) & 1) ^ 1, a.status)) return false;
      if (lane < PF_BLOCKS) vmeta[st * PF_BLOCKS + lane] = PfVMeta{d.nv, d.j0};
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], PF_TILE);
      __syncwarp();
      if (lane < PF_BLOCKS) {
        uint8_t* vd = sV + st * PF_TILE + lane * (kBlock * 128);
        tma_load_2d(vd, &vmap, &v_full[st], 0, d.y);
        tma_load_2d(vd + PF_HALF, &vmap, &v_full[st], 64, d.y);
      }
      return true;
    };
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    Lane prev{};
    for (int j = 0; j < n_tiles && ok; ++j) {
      const Lane cur = describe(j);
      ok = issue_k(j, cur);
      if (ok) k_issued = j + 1;
      if (ok && j >= 1) {
        ok = issue_v(j - 1, prev);
        if (ok) v_issued = j;
      }
      prev = cur;
    }
    if (ok && n_tiles > 0) {
      ok = issue_v(n_tiles - 1, prev);
      if (ok) v_issued = n_tiles;
    }
    if (!ok) abort_flag = 1;
    if (lane == 0) {  // every copy issued must land before the CTA exits (bounded)
      mbar_wait(q_full, 0, a.status);
      for (int j = max(0, k_issued - PF_NK); j < k_issued; ++j) mbar_wait(&k_full[j % PF_NK], (j / PF_NK) & 1, a.status);
      for (int j = max(0, v_issued - PF_NV); j < v_issued; ++j) mbar_wait(&v_full[j % PF_NV], (j / PF_NV) & 1, a.status);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(PF_BM, PF_BN, false);
      constexpr uint32_t idO = idesc_bf16_f32(PF_BM, PF_D, true);
      const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
      auto issue_s = [&](int j) {
        const uint32_t k_addr = smem_u32(sK + (j % PF_NK) * PF_TILE);
#pragma unroll
        for (int ks = 0; ks < PF_D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * PF_HALF + (ks & 3) * 32;
          tc_mma(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idS, ks > 0);
        }
        tc_commit(s_full);
        tc_commit(&k_empty[j % PF_NK]);
      };
      auto issue_pv = [&](int j) {
        const uint32_t v_addr = smem_u32(sV + (j % PF_NV) * PF_TILE);
#pragma unroll
        for (int ks = 0; ks < PF_BN / 16; ++ks) {
          const uint32_t poff = (ks >> 2) * PF_HALF + (ks & 3) * 32;
          tc_mma(tO, sdesc_sw128(p_addr + poff, 16, 1024), sdesc_sw128(v_addr + ks * 2048, PF_HALF, 1024), idO,
                 (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(pv_done);
        tc_commit(&v_empty[j % PF_NV]);
      };
      // Blocking waits (the thread sleeps instead of spinning on issue slots that
      // the softmax warps need). K runs PF_NK tiles ahead, so S(j+1) is rarely held
      // back by a load and the order S(j+1), P V(j) keeps the tensor pipe fed.
      bool ok = mbar_wait(q_ready, 0, a.status) && mbar_wait(&k_ready[0], 0, a.status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          ok = mbar_wait(&k_ready[(j + 1) % PF_NK], ((j + 1) / PF_NK) & 1, a.status) &&
               mbar_wait(s_free, j & 1, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        ok = mbar_wait(p_full, j & 1, a.status) && mbar_wait(&v_full[j % PF_NV], (j / PF_NV) & 1, a.status) &&
             mbar_wait(&v_ready[j % PF_NV], (j / PF_NV) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(j);
      }
      if (!ok) abort_flag = 1;
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- K rotation, V holes
    const int t = threadIdx.x - 128;
    const int c = t & 7, r = t >> 3;  // 16-byte chunk (8 frequencies) and row within a block
    float2 tr[8];
    Rot8 rot;
    if constexpr (LAZY) {
#pragma unroll
      for (int e = 0; e < 8; ++e) tr[e] = __ldg(&a.rope[8 * c + e]);
    }
    int p_cached = INT_MIN;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % PF_NK;
      if (!warp_wait_pf(&k_full[st], (j / PF_NK) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      uint8_t* kt = sK + st * PF_TILE;
      bool holes = false;
#pragma unroll 1
      for (int bl = 0; bl < PF_BLOCKS; ++bl) {
        const PfKMeta m = kmeta[st * PF_BLOCKS + bl];
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
            uint4 Y = *reinterpret_cast<uint4*>(kt + PF_HALF + off);
            rotate_chunk(X, Y, rot);
            *reinterpret_cast<uint4*>(kt + off) = X;
            *reinterpret_cast<uint4*>(kt + PF_HALF + off) = Y;
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&k_ready[st]);
      // V rows of hole slots may hold anything: zero them. v_ready(j) is arrived only
      // after V(j) has landed, so this warpgroup can never complete a v_ready phase
      // two tiles ahead of the MMA warp (V(j+2) needs the P V of tile j first).
      const int vs = j % PF_NV;
      if (!warp_wait_pf(&v_full[vs], (j / PF_NV) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      if (__any_sync(0xffffffffu, holes)) {
        uint8_t* vt = sV + vs * PF_TILE;
#pragma unroll 1
        for (int bl = 0; bl < PF_BLOCKS; ++bl) {
          if (r >= vmeta[vs * PF_BLOCKS + bl].nvalid) {
            const uint32_t off = bl * (kBlock * 128) + sw128(r, c);
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vt + PF_HALF + off) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&v_ready[vs]);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int i = threadIdx.x;  // query row within the tile == TMEM lane
    const int iq = row0 + i;    // query index within the chunk
    const int m_pos = a.q_start[s] + iq;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = warp_wait_pf(q_full, 0, a.status);
    if (ok) {
      // Q prologue: q_i' = R_{m_i} q_i, once per tile, pre-scaled by the softmax
      // scale * log2(e) so that S comes out of the tensor core in log2 units.
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float2 cs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) cs[e] = rope_cs(__ldg(&a.rope[8 * c + e]), m_pos, a.status);
        uint4 X = *reinterpret_cast<uint4*>(sQ + sw128(i, c));
        uint4 Y = *reinterpret_cast<uint4*>(sQ + PF_HALF + sw128(i, c));
        rotate_chunk(X, Y, make_rot8(cs, a.scale_log2));
        *reinterpret_cast<uint4*>(sQ + sw128(i, c)) = X;
        *reinterpret_cast<uint4*>(sQ + PF_HALF + sw128(i, c)) = Y;
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(q_ready);
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int vs = j % PF_NV;
      ok = warp_wait_pf(s_full, j & 1, a.status);
      if (!ok) break;
      tc_fence_after();
      float sv[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + lane_base + 32 * q, sv[q]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);
      ok = warp_wait_pf(&v_full[vs], (j / PF_NV) & 1, a.status);  // block metadata of this tile
      if (!ok) break;
      // Masks only where a tile has hole slots or chunk keys (uniform per tile).
      bool full_tile = true;
#pragma unroll
      for (int bl = 0; bl < PF_BLOCKS; ++bl) {
        const PfVMeta m = vmeta[vs * PF_BLOCKS + bl];
        full_tile &= (m.nvalid == kBlock) & (m.chunk_j0 < 0);
      }
      float mx = -INFINITY;
      if (full_tile) {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int k = 0; k < 32; k += 2) m4[q] = fmax3(m4[q], sv[q][k], sv[q][k + 1]);
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
#pragma unroll
        for (int bl = 0; bl < PF_BLOCKS; ++bl) {
          const PfVMeta m = vmeta[vs * PF_BLOCKS + bl];
          int lim = m.nvalid;
          if (m.chunk_j0 >= 0) lim = max(0, min(lim, iq - m.chunk_j0 + 1));
#pragma unroll
          for (int t = 0; t < kBlock; ++t) {
            const int kk = bl * kBlock + t;
            float& v = sv[kk >> 5][kk & 31];
            v = t < lim ? v : -INFINITY;
            mx = fmaxf(mx, v);
          }
        }
      }
      // Refresh the running maximum only when it grows by more than 2^8 (weights stay <= 256).
      float alpha = 1.f;
      if (mx > m_run + PF_RESCALE_LOG2) {
        alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
        m_run = mx;
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      // P in registers first (bf16 pairs), so that only the stores wait for the
      // previous P V product to release the buffer.
      uint32_t pw[PF_BN / 2];
      const uint64_t mm = f2(m_use, m_use);
      uint64_t acc0 = f2(0.f, 0.f), acc1 = acc0;  // row sum of the fp32 weights, packed pairs
#pragma unroll
      for (int k = 0; k < PF_BN / 2; ++k) {
        const int kk = 2 * k;
        const float2 dv = f2_split(f2_sub(f2(sv[kk >> 5][kk & 31], sv[kk >> 5][(kk + 1) & 31]), mm));
        const float e0 = ex2(dv.x), e1 = ex2(dv.y);
        pw[k] = pack_bf16x2(e0, e1);
        if (k & 1)
          acc1 = f2_add(acc1, f2(e0, e1));
        else
          acc0 = f2_add(acc0, f2(e0, e1));
      }
      const float2 sacc = f2_split(f2_add(acc0, acc1));
      l_run = l_run * alpha + (sacc.x + sacc.y);
      if (j > 0) {
        ok = warp_wait_pf(pv_done, (j - 1) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
      }
#pragma unroll
      for (int c16 = 0; c16 < PF_BN / 8; ++c16)
        *reinterpret_cast<uint4*>(sP + (c16 >> 3) * PF_HALF + sw128(i, c16 & 7)) =
            make_uint4(pw[4 * c16], pw[4 * c16 + 1], pw[4 * c16 + 2], pw[4 * c16 + 3]);
      // Rescale the running output when this row's maximum was refreshed (warp-uniform).
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(tO + lane_base + 32 * q, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tO + lane_base + 32 * q, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (!ok && n_tiles > 0) abort_flag = 1;
    // Epilogue: O / l -> bf16.
    if (ok && n_tiles > 0) ok = warp_wait_pf(pv_done, (n_tiles - 1) & 1, a.status);
    if (ok) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(q0 + iq) * a.Hq + h) * PF_D;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float o[32];
        if (n_tiles > 0) {
          tmem_ld32(tO + lane_base + 32 * q, o);
          tmem_ld_wait();
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
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, PF_TMEM_COLS);
  }
}

cudaError_t launch_prefill(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t st) {
  if (a.D != PF_D) return cudaErrorNotSupported;
  if (a.B == 0 || a.max_q_len == 0) return cudaSuccess;
#ifndef LAZY_PREFILL_SINGLE_TILE
  if (a.G % 2 == 0) return launch_prefill_pair(a, lazy, qmap, kmap, vmap, st);
#endif
  dim3 grid((a.max_q_len + PF_BM - 1) / PF_BM, a.Hq, a.B);
  auto kern = lazy ? prefill_kernel<true> : prefill_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, PF_THREADS, PF_SMEM, st>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace lazy
