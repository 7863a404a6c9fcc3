// decode_f32.cu -- LazyAttention decode for fp32 pools (plain SIMT, exact-ish fp32).
//
// Same contract as the bf16 kernel ("Resumo Técnico: LazyAttention",
// "Implementação Técnica", item 2): the query of each head is re-rotated by
// R_{m-p} only when the document start p changes, keys are read as stored, and
// an online (max, sum) softmax runs over the 16-token blocks. This path exists
// for fp32 caches (small models, tests); it keeps every product in fp32.
//
// CTA = (split, KV head, sequence), 128 threads; warp w owns q-heads
// w, w+4, ... of the group. Each block's K and V rows are staged in shared
// memory; lane t < 16 scores key t, lanes own output columns lane + 32j.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace lazy {

constexpr int kF32Threads = 128;
constexpr int kF32MaxHeadsPerWarp = 8;  // g <= 32

template <int D, bool LAZY>
__global__ void __launch_bounds__(kF32Threads) decode_f32_kernel(const DecodeArgs a) {
  constexpr int HALF = D / 2, PER = D / 32;
  extern __shared__ float sm[];
  float* Ks = sm;                   // [16][D]
  float* Vs = Ks + kBlock * D;      // [16][D]
  float* qraw = Vs + kBlock * D;    // [G][D]
  float* qrot = qraw + a.G * D;     // [G][D]
  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const int b0 = split * a.bps, b1 = min(nb, b0 + a.bps);
  const int m_pos = a.q_pos[s];
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;
  const float* kp = static_cast<const float*>(a.k_pool);
  const float* vp = static_cast<const float*>(a.v_pool);
  const float* qg = static_cast<const float*>(a.q) + ((size_t)s * a.Hq + (size_t)kvh * a.G) * D;
  for (int i = threadIdx.x; i < a.G * D; i += kF32Threads) qraw[i] = qg[i];
  __syncthreads();

  float m_r[kF32MaxHeadsPerWarp], l_r[kF32MaxHeadsPerWarp], o[kF32MaxHeadsPerWarp][PER];
#pragma unroll
  for (int hh = 0; hh < kF32MaxHeadsPerWarp; ++hh) {
    m_r[hh] = -INFINITY;
    l_r[hh] = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) o[hh][j] = 0.f;
  }
  // Rotate this warp's heads by R_delta into qrot.
  auto rotate = [&](int delta) {
    for (int h = warp; h < a.G; h += 4)
      for (int i = lane; i < HALF; i += 32) {
        const float2 c = rope_cs(__ldg(&a.rope[i]), delta, a.status);
        const float x = qraw[h * D + i], y = qraw[h * D + i + HALF];
        qrot[h * D + i] = fmaf(x, c.x, -y * c.y);
        qrot[h * D + i + HALF] = fmaf(y, c.x, x * c.y);
      }
    __syncwarp();
  };
  if (!LAZY) rotate(m_pos);
  int p_prev = INT_MIN;
  for (int b = b0; b < b1; ++b) {
    const BlockInfo bi = decode_word(__ldg(&wrow[b]), b, a.id_bits);
    const int p_next = b + 1 < nb ? decode_word(__ldg(&wrow[b + 1]), b + 1, a.id_bits).p : bi.p;
    int nvalid = block_valid(b, nb, seq_len, bi.p, p_next);
    nvalid = nvalid < 0 ? 0 : (nvalid > kBlock ? kBlock : nvalid);
    const bool ok = bi.phys < a.num_pool_blocks;
    if (!ok) {
      nvalid = 0;
      if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
    }
    __syncthreads();  // previous block's rows are no longer read
    const size_t base = ((size_t)(ok ? bi.phys : 0) * a.Hkv + kvh) * kBlock * D;
    for (int i = threadIdx.x; i < kBlock * D; i += kF32Threads) {
      const bool v = ok && (i / D) < nvalid;
      Ks[i] = v ? kp[base + i] : 0.f;
      Vs[i] = v ? vp[base + i] : 0.f;
    }
    __syncthreads();
    if (LAZY && bi.p != p_prev) {
      rotate(m_pos - bi.p);
      p_prev = bi.p;
    }
#pragma unroll
    for (int hh = 0; hh < kF32MaxHeadsPerWarp; ++hh) {
      const int h = warp + 4 * hh;
      if (h >= a.G) break;
      float sc = -INFINITY;
      if (lane < nvalid) {
        float acc = 0.f;
        for (int c = 0; c < D; ++c) acc = fmaf(qrot[h * D + c], Ks[lane * D + c], acc);
        sc = acc * a.scale_log2;
      }
      float mx = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m_r[hh], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = exp2f(m_r[hh] - m_use);
      const float pj = exp2f(sc - m_use);
      float ps = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      m_r[hh] = m_new;
      l_r[hh] = l_r[hh] * alpha + ps;
#pragma unroll
      for (int j = 0; j < PER; ++j) o[hh][j] *= alpha;
      for (int t = 0; t < kBlock; ++t) {
        const float pt = __shfl_sync(0xffffffffu, pj, t);
#pragma unroll
        for (int j = 0; j < PER; ++j) o[hh][j] = fmaf(pt, Vs[t * D + lane + 32 * j], o[hh][j]);
      }
    }
  }
#pragma unroll
  for (int hh = 0; hh < kF32MaxHeadsPerWarp; ++hh) {
    const int h = warp + 4 * hh;
    if (h >= a.G) break;
    const int hq = kvh * a.G + h;
    if (a.splits == 1) {
      const float inv = l_r[hh] > 0.f ? 1.f / l_r[hh] : 0.f;
      float* dst = static_cast<float*>(a.out) + ((size_t)s * a.Hq + hq) * D;
#pragma unroll
      for (int j = 0; j < PER; ++j) dst[lane + 32 * j] = o[hh][j] * inv;
    } else {
      const size_t pidx = ((size_t)s * a.Hq + hq) * a.splits + split;
#pragma unroll
      for (int j = 0; j < PER; ++j) a.ws_o[pidx * D + lane + 32 * j] = o[hh][j];
      if (lane == 0) {
        a.ws_ml[2 * pidx] = m_r[hh];
        a.ws_ml[2 * pidx + 1] = l_r[hh];
      }
    }
  }
}

cudaError_t launch_decode_f32(const DecodeArgs& a, bool lazy, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.B);
  const int smem = (2 * kBlock * a.D + 2 * a.G * a.D) * (int)sizeof(float);
  cudaError_t e;
  if (a.D == 128) {
    auto k = lazy ? decode_f32_kernel<128, true> : decode_f32_kernel<128, false>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    k<<<grid, kF32Threads, smem, st>>>(a);
  } else {
    auto k = lazy ? decode_f32_kernel<64, true> : decode_f32_kernel<64, false>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
    k<<<grid, kF32Threads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

// fp32 debug gather: the same word decode and hole rule with plain loads.
__global__ void gather_f32_kernel(const GatherArgs a) {
  const int kvh = blockIdx.x, s = blockIdx.y;
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const uint32_t* wrow = a.words + (size_t)s * a.max_blocks;
  const size_t rows = (size_t)kBlock * a.max_blocks;
  float* kout = static_cast<float*>(a.k_out) + ((size_t)s * a.Hkv + kvh) * rows * a.D;
  float* vout = static_cast<float*>(a.v_out) + ((size_t)s * a.Hkv + kvh) * rows * a.D;
  const float* kp = static_cast<const float*>(a.k_pool);
  const float* vp = static_cast<const float*>(a.v_pool);
  for (int b = 0; b < a.max_blocks; ++b) {
    int nvalid = 0, p = -1, phys = 0;
    if (b < nb) {
      const BlockInfo bi = decode_word(__ldg(&wrow[b]), b, a.id_bits);
      const int p_next = b + 1 < nb ? decode_word(__ldg(&wrow[b + 1]), b + 1, a.id_bits).p : bi.p;
      nvalid = block_valid(b, nb, seq_len, bi.p, p_next);
      nvalid = nvalid < 0 ? 0 : (nvalid > kBlock ? kBlock : nvalid);
      p = bi.p;
      phys = bi.phys;
      if (phys >= a.num_pool_blocks) {
        nvalid = 0;
        if (threadIdx.x == 0) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
      }
    }
    const size_t base = ((size_t)phys * a.Hkv + kvh) * kBlock * a.D;
    for (int i = threadIdx.x; i < kBlock * a.D; i += blockDim.x) {
      const bool v = (i / a.D) < nvalid;
      kout[(size_t)kBlock * b * a.D + i] = v ? kp[base + i] : 0.f;
      vout[(size_t)kBlock * b * a.D + i] = v ? vp[base + i] : 0.f;
    }
    if (a.pos_out && kvh == 0 && threadIdx.x < kBlock)
      a.pos_out[(size_t)s * rows + kBlock * b + threadIdx.x] = (int)threadIdx.x < nvalid ? p : -1;
  }
}

cudaError_t launch_gather_f32(const GatherArgs& a, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  gather_f32_kernel<<<dim3(a.Hkv, a.B), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lazy
