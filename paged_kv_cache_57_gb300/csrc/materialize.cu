// materialize.cu -- the eager, position-materialising alternative to LazyAttention.
//
// "Declaração do Problema" (technical summary "Resumo Técnico: LazyAttention"):
// without lazy positions, a cached document reused at a new offset p must have its
// keys re-rotated to their absolute positions before standard attention can read
// them, and each sequence then owns its own copy. This kernel does exactly that for
// a batch: every logical block b of every sequence s gets a private block
// s * max_blocks + b in an output pool, holding K rotated by R_p (stored K already
// carries its document-local position j, so R_p R_j k = R_{p+j} k) and V copied.
// The output block words point at the copies and keep the offset field, so the
// control path of lazy_attn_decode (lazy = 0: q rotated once by R_m, no per-document
// rotation) reads them. It exists to measure what the lazy method avoids: the copy
// traffic, the per-sequence footprint, and a decode that cannot share blocks.
//
// One warp per (sequence, logical block, KV head): lane l handles 16-byte chunk
// c = l % (D/16) of the row pairs (i, i + D/2); the chunk's 8 frequencies'
// (cos, sin) of p * w_f are evaluated once per block in registers.
#include "common.cuh"
#include "kernels.h"

namespace lazy {

template <int D>
__global__ void __launch_bounds__(256) materialize_kernel(const MaterializeArgs a) {
  constexpr int HALF = D / 2, CH = HALF / 8;  // 16-byte chunks per half row
  constexpr int ROWS_PER_PASS = 32 / CH;
  const long long task = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long ntask = (long long)a.B * a.max_blocks * a.Hkv;
  if (task >= ntask) return;
  const int kvh = (int)(task % a.Hkv);
  const long long sb = task / a.Hkv;
  const int s = (int)(sb / a.max_blocks), b = (int)(sb % a.max_blocks);
  int seq_len = a.seq_lens[s];
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    if (lane == 0 && kvh == 0) raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  const int nb = (seq_len + kBlock - 1) / kBlock;
  const uint32_t w = a.words[(size_t)s * a.max_blocks + b];
  const size_t dst_block = (size_t)s * a.max_blocks + b;
  if (kvh == 0 && lane == 0) {
    // The copy's word: same offset field (so p and the hole rule decode unchanged), new id.
    const uint32_t id_mask = (1u << a.id_bits) - 1u;
    a.words_out[dst_block] = b < nb ? ((w & ~id_mask) | ((uint32_t)dst_block & id_mask)) : 0u;
  }
  if (b >= nb) return;
  const BlockInfo bi = decode_word(w, b, a.id_bits);
  if (bi.phys >= a.num_pool_blocks) {
    if (lane == 0) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
    return;
  }
  const int c = lane % CH;
  float2 cs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) cs[e] = rope_cs(__ldg(&a.rope[8 * c + e]), bi.p, a.status);
  const size_t src_off = ((size_t)bi.phys * a.Hkv + kvh) * kBlock * D;
  const size_t dst_off = (dst_block * a.Hkv + kvh) * kBlock * D;
  const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.k_pool) + src_off);
  const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v_pool) + src_off);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.k_out) + dst_off);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.v_out) + dst_off);
  // V: a plain copy of the block, 16 bytes per lane per step.
  for (int idx = lane; idx < kBlock * D / 8; idx += 32) vd[idx] = __ldg(&vs[idx]);
  // K: rows r, chunk c of both halves; x' = x cos - y sin, y' = y cos + x sin in fp32.
  for (int r = lane / CH; r < kBlock; r += ROWS_PER_PASS) {
    const uint4 X = __ldg(&ks[r * (D / 8) + c]);
    const uint4 Y = __ldg(&ks[r * (D / 8) + CH + c]);
    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&X);
    const uint32_t* yw = reinterpret_cast<const uint32_t*>(&Y);
    uint4 Xo, Yo;
    uint32_t* xo = reinterpret_cast<uint32_t*>(&Xo);
    uint32_t* yo = reinterpret_cast<uint32_t*>(&Yo);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x0 = __uint_as_float(xw[k] << 16), x1 = __uint_as_float(xw[k] & 0xffff0000u);
      const float y0 = __uint_as_float(yw[k] << 16), y1 = __uint_as_float(yw[k] & 0xffff0000u);
      const float2 c0 = cs[2 * k], c1 = cs[2 * k + 1];
      xo[k] = pack_bf16x2(fmaf(x0, c0.x, -y0 * c0.y), fmaf(x1, c1.x, -y1 * c1.y));
      yo[k] = pack_bf16x2(fmaf(y0, c0.x, x0 * c0.y), fmaf(y1, c1.x, x1 * c1.y));
    }
    kd[r * (D / 8) + c] = Xo;
    kd[r * (D / 8) + CH + c] = Yo;
  }
}

cudaError_t launch_materialize(const MaterializeArgs& a, cudaStream_t st) {
  const long long ntask = (long long)a.B * a.max_blocks * a.Hkv;
  if (ntask == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (ntask + 7) / 8;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  if (a.D == 128)
    materialize_kernel<128><<<(unsigned)blocks, threads, 0, st>>>(a);
  else
    materialize_kernel<64><<<(unsigned)blocks, threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lazy
