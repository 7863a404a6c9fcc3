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
//   warps 0-3  softmax: rotate the Q tile once (thread = row), then per K tile
//              read S from TMEM, mask (holes; causal inside the chunk), online
//              (max, sum) softmax ("Flash Attention -- tiling"), write P (bf16,
//              128-byte swizzled K-major) to shared memory, rescale O in TMEM;
//              finally O / l -> bf16 -> global.
//   warps 4-7  rotation: rotate every 16-row K block of a landed tile in shared
//              memory by R_p (fp32 math, bf16 result) and zero V rows of hole
//              slots, then hand the tile to the MMA warp.
//   warp 8     TMA producer: Q tile, then per tile 8 blocks x (K, V) x 2 boxes
//              of 16 rows x 64 columns, into a ring of PF_NS stages.
//   warp 9     TMEM owner and MMA issuer: S = Q K^T (M=N=128, K=d) into TMEM
//              columns [0,128), O += P V into columns [128,256); S of the next
//              tile is issued while the softmax works on the current one.
#include <climits>

#include "kernels.h"
#include "tcgen05.cuh"

namespace lazy {

namespace {

constexpr int PF_BM = 128;                      // query rows per tile (MMA M)
constexpr int PF_BN = 128;                      // keys per tile (MMA N of S)
constexpr int PF_D = 128;                       // head dim
constexpr int PF_NS = 2;                        // K/V stages
constexpr int PF_BLOCKS = PF_BN / kBlock;       // 8 blocks per key tile
constexpr int PF_HALF = PF_BM * 128;            // one 64-column half of a 128-row tile (bytes)
constexpr int PF_TILE = 2 * PF_HALF;            // 32 KiB
constexpr int PF_THREADS = 320;
constexpr int PF_TMEM_COLS = 256;

struct PfBlockMeta {
  int p;         // document start position
  int nvalid;    // valid slots (0 for blocks past the sequence or with a bad id)
  int chunk_j0;  // chunk-local index of the block's first key, or -1 for cached documents
  int pad;
};

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + PF_TILE;
constexpr int OFF_V = OFF_K + PF_NS * PF_TILE;
constexpr int OFF_P = OFF_V + PF_NS * PF_TILE;
constexpr int OFF_META = OFF_P + PF_TILE;
constexpr int OFF_BAR = OFF_META + PF_NS * PF_BLOCKS * (int)sizeof(PfBlockMeta);
constexpr int NBARS = 2 + 3 * PF_NS + 5;
constexpr int OFF_TMEM = OFF_BAR + NBARS * 8;
constexpr int PF_SMEM = 1024 + OFF_TMEM + 16;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool warp_wait_pf(uint64_t* bar, uint32_t parity, unsigned int* status) {
  const bool ok = mbar_wait(bar, parity, status);
  return __all_sync(0xffffffffu, ok);
}

// Rotates 8 rotate-half pairs held as two 16-byte chunks (x: dims i, y: dims i + 64).
__device__ __forceinline__ void rotate_chunk(uint4& X, uint4& Y, const float2 (&cs)[8]) {
  uint32_t* xw = reinterpret_cast<uint32_t*>(&X);
  uint32_t* yw = reinterpret_cast<uint32_t*>(&Y);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[k]));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&yw[k]));
    const float2 c0 = cs[2 * k], c1 = cs[2 * k + 1];
    const float x0 = fmaf(x.x, c0.x, -y.x * c0.y), y0 = fmaf(y.x, c0.x, x.x * c0.y);
    const float x1 = fmaf(x.y, c1.x, -y.y * c1.y), y1 = fmaf(y.y, c1.x, x.y * c1.y);
    xw[k] = pack_bf16x2(x0, x1);
    yw[k] = pack_bf16x2(y0, y1);
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
  PfBlockMeta* meta = reinterpret_cast<PfBlockMeta*>(base + OFF_META);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_ready = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_ready = kv_full + PF_NS;
  uint64_t* kv_empty = kv_ready + PF_NS;
  uint64_t* s_full = kv_empty + PF_NS;
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
    for (int i = 0; i < PF_NS; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_ready[i], 128);
      mbar_init(&kv_empty[i], 1);
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
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % PF_NS;
      if (j >= PF_NS && !warp_wait_pf(&kv_empty[st], ((j / PF_NS) & 1) ^ 1, a.status)) {
        abort_flag = 1;
        break;
      }
      // lanes 0..7: the tile's blocks; lane 8: the block after (hole rule)
      const int b = j * PF_BLOCKS + min(lane, PF_BLOCKS);
      const uint32_t w = (lane <= PF_BLOCKS && b < nb) ? __ldg(&wrow[b]) : 0u;
      const BlockInfo bi = decode_word(w, b, a.id_bits);
      const int p_after = __shfl_down_sync(0xffffffffu, bi.p, 1);
      int nv = 0, y = -kBlock, j0 = -1;
      if (lane < PF_BLOCKS && b < nb) {
        nv = block_valid(b, nb, seq_len, bi.p, b + 1 < nb ? p_after : bi.p);
        nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
        if (bi.phys < a.num_pool_blocks) {
          y = (bi.phys * a.Hkv + kvh) * kBlock;
        } else {
          raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
          nv = 0;
        }
        j0 = b >= b_chunk ? kBlock * (b - b_chunk) : -1;
      }
      if (lane < PF_BLOCKS) meta[st * PF_BLOCKS + lane] = PfBlockMeta{bi.p, nv, j0, 0};
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], 2 * PF_TILE);
      __syncwarp();
      if (lane < PF_BLOCKS) {  // rows of an invalid block start at -16: read as zeros
        uint8_t* kd = sK + st * PF_TILE + lane * (kBlock * 128);
        uint8_t* vd = sV + st * PF_TILE + lane * (kBlock * 128);
        tma_load_2d(kd, &kmap, &kv_full[st], 0, y);
        tma_load_2d(kd + PF_HALF, &kmap, &kv_full[st], 64, y);
        tma_load_2d(vd, &vmap, &kv_full[st], 0, y);
        tma_load_2d(vd + PF_HALF, &vmap, &kv_full[st], 64, y);
      }
      issued = j + 1;
    }
    if (lane == 0) {
      mbar_wait(q_full, 0, a.status);
      for (int j = max(0, issued - PF_NS); j < issued; ++j)
        mbar_wait(&kv_full[j % PF_NS], (j / PF_NS) & 1, a.status);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(PF_BM, PF_BN, false);
      constexpr uint32_t idO = idesc_bf16_f32(PF_BM, PF_D, true);
      const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
      auto issue_S = [&](int j) {
        const uint32_t k_addr = smem_u32(sK + (j % PF_NS) * PF_TILE);
#pragma unroll
        for (int ks = 0; ks < PF_D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * PF_HALF + (ks & 3) * 32;
          tc_mma(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idS, ks > 0);
        }
        tc_commit(s_full);
      };
      auto issue_PV = [&](int j) {
        const uint32_t v_addr = smem_u32(sV + (j % PF_NS) * PF_TILE);
#pragma unroll
        for (int ks = 0; ks < PF_BN / 16; ++ks) {
          const uint32_t poff = (ks >> 2) * PF_HALF + (ks & 3) * 32;
          tc_mma(tO, sdesc_sw128(p_addr + poff, 16, 1024), sdesc_sw128(v_addr + ks * 2048, PF_HALF, 1024), idO,
                 (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(pv_done);
        tc_commit(&kv_empty[j % PF_NS]);
      };
      bool ok = n_tiles > 0 && mbar_wait(q_ready, 0, a.status) && mbar_wait(&kv_ready[0], 0, a.status);
      if (ok) {
        tc_fence_after();
        issue_S(0);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
          ok = mbar_wait(&kv_ready[(j + 1) % PF_NS], ((j + 1) / PF_NS) & 1, a.status) &&
               mbar_wait(s_free, j & 1, a.status);
          if (!ok) break;
          tc_fence_after();
          issue_S(j + 1);
        }
        ok = mbar_wait(p_full, j & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        issue_PV(j);
      }
      if (!ok && n_tiles > 0) abort_flag = 1;
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- K rotation
    const int t = threadIdx.x - 128;
    const int c = t & 7, r = t >> 3;  // 16-byte chunk (8 frequencies) and row within a block
    float2 tr[8], cs[8];
    if constexpr (LAZY) {
#pragma unroll
      for (int e = 0; e < 8; ++e) tr[e] = __ldg(&a.rope[8 * c + e]);
    }
    int p_cached = INT_MIN;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % PF_NS;
      if (!warp_wait_pf(&kv_full[st], (j / PF_NS) & 1, a.status)) {
        abort_flag = 1;
        break;
      }
      uint8_t* kt = sK + st * PF_TILE;
      uint8_t* vt = sV + st * PF_TILE;
#pragma unroll 1
      for (int bl = 0; bl < PF_BLOCKS; ++bl) {
        const PfBlockMeta m = meta[st * PF_BLOCKS + bl];
        const uint32_t off = bl * (kBlock * 128) + sw128(r, c);
        if constexpr (LAZY) {
          if (m.nvalid > 0) {
            if (m.p != p_cached) {
#pragma unroll
              for (int e = 0; e < 8; ++e) cs[e] = rope_cs(tr[e], m.p, a.status);
              p_cached = m.p;
            }
            uint4 X = *reinterpret_cast<uint4*>(kt + off);
            uint4 Y = *reinterpret_cast<uint4*>(kt + PF_HALF + off);
            rotate_chunk(X, Y, cs);
            *reinterpret_cast<uint4*>(kt + off) = X;
            *reinterpret_cast<uint4*>(kt + PF_HALF + off) = Y;
          }
        }
        if (r >= m.nvalid) {  // hole slot: its V row may hold anything
          *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vt + PF_HALF + off) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&kv_ready[st]);
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int i = threadIdx.x;        // query row within the tile == TMEM lane
    const int iq = row0 + i;          // query index within the chunk
    const int m_pos = a.q_start[s] + iq;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = warp_wait_pf(q_full, 0, a.status);
    if (ok) {
      // Q prologue: q_i' = R_{m_i} q_i, once per tile.
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float2 cs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) cs[e] = rope_cs(__ldg(&a.rope[8 * c + e]), m_pos, a.status);
        uint4 X = *reinterpret_cast<uint4*>(sQ + sw128(i, c));
        uint4 Y = *reinterpret_cast<uint4*>(sQ + PF_HALF + sw128(i, c));
        rotate_chunk(X, Y, cs);
        *reinterpret_cast<uint4*>(sQ + sw128(i, c)) = X;
        *reinterpret_cast<uint4*>(sQ + PF_HALF + sw128(i, c)) = Y;
      }
      fence_proxy_async_smem();
    }
    mbar_arrive(q_ready);
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int st = j % PF_NS;
      ok = warp_wait_pf(s_full, j & 1, a.status);
      if (!ok) break;
      tc_fence_after();
      float sv[4][32];
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(tS + lane_base + 32 * q, sv[q]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);
      ok = warp_wait_pf(&kv_full[st], (j / PF_NS) & 1, a.status);  // block metadata of this tile
      if (!ok) break;
      float mx = -INFINITY;
#pragma unroll
      for (int bl = 0; bl < PF_BLOCKS; ++bl) {
        const PfBlockMeta m = meta[st * PF_BLOCKS + bl];
        int lim = m.nvalid;
        if (m.chunk_j0 >= 0) lim = max(0, min(lim, iq - m.chunk_j0 + 1));
#pragma unroll
        for (int t = 0; t < kBlock; ++t) {
          const int kk = bl * kBlock + t;
          float& v = sv[kk >> 5][kk & 31];
          v = t < lim ? v * sl2 : -INFINITY;
          mx = fmaxf(mx, v);
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      m_run = m_new;
      // P: wait until the previous P V product has consumed the buffer.
      if (j > 0) {
        ok = warp_wait_pf(pv_done, (j - 1) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
      }
      float sum = 0.f;
#pragma unroll
      for (int c16 = 0; c16 < PF_BN / 8; ++c16) {
        uint32_t wds[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int kk = c16 * 8 + 2 * k;
          const uint32_t pk = pack_bf16x2(exp2f(sv[kk >> 5][kk & 31] - m_use), exp2f(sv[kk >> 5][(kk + 1) & 31] - m_use));
          const float2 back = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk));
          sum += back.x + back.y;
          wds[k] = pk;
        }
        *reinterpret_cast<uint4*>(sP + (c16 >> 3) * PF_HALF + sw128(i, c16 & 7)) =
            make_uint4(wds[0], wds[1], wds[2], wds[3]);
      }
      l_run = l_run * alpha + sum;
      // Rescale the running output when this row's maximum grew (warp-uniform).
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
  dim3 grid((a.max_q_len + PF_BM - 1) / PF_BM, a.Hq, a.B);
  auto kern = lazy ? prefill_kernel<true> : prefill_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PF_SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, PF_THREADS, PF_SMEM, st>>>(a, qmap, kmap, vmap);
  return cudaGetLastError();
}

}  // namespace lazy
