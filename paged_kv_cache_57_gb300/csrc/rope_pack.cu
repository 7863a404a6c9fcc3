// rope_pack.cu -- rotation table initialisation and the device block-word packer.
#include "common.cuh"
#include "kernels.h"

namespace lazy {

// t_i = w_i / (2 pi), w_i = theta^(-2i/d) (with the Llama-3.1 wavelength-band scaling
// of lazy_attn.h when requested), in fp64, stored as fp32 (hi, lo).
// Entries [0, half): the turns (hi, lo). Entries half + i * half + f: (cos, sin)(i w_f)
// for the prefill row offsets i < LAZY_ROPE_ROWS. Everything in fp64, rounded once.
// Scaling parameters of the frequencies; factor <= 0 means none.
struct FreqScale {
  double factor, low_ff, high_ff, orig_max;
};
// Explicit rates (radians per position), passed by value; `on` selects them.
struct ExplicitRates {
  double w[64];
  int on;
};

__global__ void rope_table_kernel(float2* table, int half, int head_dim, double theta, FreqScale sc,
                                  ExplicitRates ex) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= half * (1 + LAZY_ROPE_ROWS)) return;
  const int f = idx % half, row = idx / half - 1;
  const double two_pi = 6.283185307179586476925286766559;
  double w = ex.on ? ex.w[f] : pow(theta, -2.0 * (double)f / (double)head_dim);
  if (!ex.on && sc.factor > 0.0) {  // wavelength bands: keep, divide by the factor, or blend the two
    const double lam = two_pi / w;
    const double lam_short = sc.orig_max / sc.high_ff, lam_long = sc.orig_max / sc.low_ff;
    if (lam > lam_long) {
      w = w / sc.factor;
    } else if (lam >= lam_short) {
      const double blend = (sc.orig_max / lam - sc.low_ff) / (sc.high_ff - sc.low_ff);
      w = (1.0 - blend) * (w / sc.factor) + blend * w;
    }
  }
  if (row < 0) {
    const double t = w / two_pi;
    const float hi = (float)t;
    table[idx] = make_float2(hi, (float)(t - (double)hi));
  } else {
    double sn, cs;
    sincos((double)row * w, &sn, &cs);
    table[idx] = make_float2((float)cs, (float)sn);
  }
}

cudaError_t launch_rope_table(float2* table, int head_dim, double theta, const lazy_rope_scaling* scaling,
                              const double* explicit_w, cudaStream_t st) {
  const int half = head_dim / 2;
  if (half > 64) return cudaErrorInvalidValue;
  const int total = half * (1 + LAZY_ROPE_ROWS);
  FreqScale sc{0.0, 1.0, 2.0, 1.0};
  if (scaling) sc = FreqScale{scaling->factor, scaling->low_freq_factor, scaling->high_freq_factor,
                              (double)scaling->original_max_position};
  ExplicitRates ex{};
  if (explicit_w) {
    ex.on = 1;
    for (int f = 0; f < half; ++f) ex.w[f] = explicit_w[f];
  }
  rope_table_kernel<<<(total + 255) / 256, 256, 0, st>>>(table, half, head_dim, theta, sc, ex);
  return cudaGetLastError();
}

__global__ void debug_rope_kernel(const float2* __restrict__ table, const int32_t* __restrict__ deltas, int n, int half,
                                  float2* out, unsigned int* status) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n * half) return;
  out[idx] = rope_cs(table[idx % half], deltas[idx / half], status);
}

cudaError_t launch_debug_rope(const float2* table, const int32_t* deltas, int n, int head_dim, float2* out,
                              unsigned int* status, cudaStream_t st) {
  const int total = n * (head_dim / 2);
  if (total == 0) return cudaSuccess;
  debug_rope_kernel<<<(total + 255) / 256, 256, 0, st>>>(table, deltas, n, head_dim / 2, out, status);
  return cudaGetLastError();
}

// One warp per sequence. Segments are taken 32 at a time: each lane checks one
// segment, an inclusive warp scan gives every segment its first logical block
// and start position, then the warp writes the words of those segments.
__global__ void pack_words_kernel(const PackArgs a) {
  const int warps_per_cta = blockDim.x >> 5;
  const int s = blockIdx.x * warps_per_cta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (s >= a.B) return;
  const int k0 = a.seg_indptr[s], k1 = a.seg_indptr[s + 1];
  const uint32_t id_mask = (1u << a.id_bits) - 1u;
  const int off_lo = -(1 << (31 - a.id_bits)), off_hi = (1 << (31 - a.id_bits)) - 1;
  uint32_t* wrow = a.words + (size_t)s * a.max_blocks;
  int blk = 0;                                 // first logical block of the next chunk
  long long pos = a.seq_pos0 ? a.seq_pos0[s] : 0;  // start position of the next chunk
  int last_len = 0;
  bool bad = (k1 < k0);
  for (int kb = k0; kb < k1 && !bad; kb += 32) {
    const int k = kb + lane;
    const bool live = k < k1;
    int len = 0, nbk = 0, doc = 0;
    bool err = false;
    if (live) {
      doc = a.seg_doc[k];
      len = a.seg_len[k];
      err = doc < 0 || doc >= a.num_docs || len < 1;
      if (!err) {
        const int dblk = a.doc_block_indptr[doc + 1] - a.doc_block_indptr[doc];
        err = len > kBlock * dblk;
        nbk = (len + kBlock - 1) / kBlock;
      }
    }
    // inclusive scans of blocks and tokens
    int sb = nbk;
    long long sp = len;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int tb = __shfl_up_sync(0xffffffffu, sb, off);
      const long long tp = __shfl_up_sync(0xffffffffu, sp, off);
      if (lane >= off) sb += tb, sp += tp;
    }
    const int my_blk = blk + sb - nbk;
    const long long my_pos = pos + sp - len;
    bad = __any_sync(0xffffffffu, err) || (blk + __shfl_sync(0xffffffffu, sb, 31) > a.max_blocks);
    if (bad) break;
    // every segment of this chunk, lanes over its blocks
    const int nlive = min(32, k1 - kb);
    for (int j = 0; j < nlive; ++j) {
      const int dj = __shfl_sync(0xffffffffu, doc, j);
      const int bj = __shfl_sync(0xffffffffu, my_blk, j);
      const long long pj = __shfl_sync(0xffffffffu, my_pos, j);
      const int nj = __shfl_sync(0xffffffffu, nbk, j);
      const int* ids = a.doc_blocks + a.doc_block_indptr[dj];
      bool e2 = false;
      for (int q = lane; q < nj; q += 32) {
        const int phys = ids[q];
        const long long off = (long long)kBlock * (bj + q) - pj - (a.key_positions ? (long long)kBlock * q : 0);
        e2 |= phys < 0 || phys >= a.num_pool_blocks || (uint32_t)phys > id_mask || off < off_lo || off > off_hi;
        wrow[bj + q] = ((uint32_t)(int)off << a.id_bits) | ((uint32_t)phys & id_mask);
      }
      bad |= __any_sync(0xffffffffu, e2);
    }
    last_len = __shfl_sync(0xffffffffu, len, nlive - 1);
    blk += __shfl_sync(0xffffffffu, sb, 31);
    pos += __shfl_sync(0xffffffffu, sp, 31);
  }
  if (bad) {
    if (lane == 0) {
      raise_status(a.status, LAZY_DEV_LAYOUT);
      a.seq_lens[s] = 0;
    }
    for (int b = lane; b < a.max_blocks; b += 32) wrow[b] = 0u;
    return;
  }
  for (int b = blk + lane; b < a.max_blocks; b += 32) wrow[b] = 0u;
  if (lane == 0) {
    const int last_blocks = (last_len + kBlock - 1) / kBlock;
    a.seq_lens[s] = blk == 0 ? 0 : kBlock * blk - (kBlock * last_blocks - last_len);
  }
}

cudaError_t launch_pack(const PackArgs& a, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  const int warps = 4;
  pack_words_kernel<<<(a.B + warps - 1) / warps, 32 * warps, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace lazy
