// prefill_stream.cu -- LazyAttention prefill, two query tiles per CTA, persistent
// stream-K schedule (sm_103a).
//
// The method ("Resumo Técnico: LazyAttention", "Implementação Técnica", item 1):
// Q rotated once by R_m per row; each 16-row K block rotated once by R_p of its
// document in shared memory (one relative rotation per K tile, no unrotate
// pass); S = Q'K^T and O += P V on tcgen05 with fp32 accumulators in TMEM.
//
// Work unit u = (sequence s, 128-row query tile, q-head pair hp): q-heads 2hp and
// 2hp+1 share one KV head (even GQA ratio), so every loaded and rotated K/V tile
// serves 2 x 128 query rows. A unit needs n(u) K tiles of 128 keys. The launch has
// one CTA per SM; the flattened sequence of (unit, K tile) iterations is cut into
// equal contiguous ranges, one per CTA (stream-K), so no SM idles at the end of a
// wave. A CTA walks its range as segments (u, tiles j0..j1-1). A unit cut by a
// range boundary is computed in pieces by consecutive CTAs: every piece writes an
// fp32 partial (o, m, l) per query row, and the thread of the last piece to finish
// a row (an arrival counter per row) merges that row's pieces with the
// online-softmax rescale and writes the output. Nothing waits on another CTA.
//
//   warps 0-3   tile A, warps 4-7 tile B (thread = query row = TMEM lane): per
//               segment R_m of the row of Q (angle addition from per-segment angles
//               of the 16-row multiples); softmax: S read from TMEM in 32-column
//               chunks twice (row maximum, then weights); P written back as bf16
//               over the tile's S columns (A operand of P V from TMEM), the first 64
//               keys' P handed over before the rest; the next K tile's key masks
//               read right after (shared-memory loads wait long while the S
//               products stream their operands); epilogue.
//   warps 8-11  per K tile, R_p of each 16-row block and V hole zeroing.
//   warp 12     TMA producer of Q and the K ring; warp 14 of the V ring. A tile is
//               16 boxes of 16 rows x 64 columns issued by 16 lanes.
//   warp 13     TMEM owner (512 columns: S_A/P_A, S_B/P_B, O_A, O_B) and MMA issuer.
// Every ring and buffer is tracked with CTA-wide counters (tiles g, segments sg),
// so the pipeline runs on across segment boundaries: the producers load the next
// segment's Q and K/V tiles while the current one drains.
#include <climits>
#include <type_traits>

#include "prefill_common.cuh"

namespace lazy {

namespace {

using namespace pf;

constexpr int NK = 2, NV = 2;

// Rotation coefficients (cos, sin) (p w_f) of frequencies 8 c .. 8 c + 7, for a K block
// at position p (the table's first D / 2 entries are the frequencies in turns). Out of
// line: the position changes only at document boundaries.
__device__ __noinline__ Rot8 block_rot8(const float2* __restrict__ rope, int c, int p, unsigned int* status) {
  float2 cs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) cs[e] = rope_cs(__ldg(&rope[8 * c + e]), p, status);
  return make_rot8(cs, 1.f);
}

constexpr int THREADS = 480;  // 15 warps
// A tile's fp32 partial: 33 column groups x 128 rows x 4 floats (groups 0..31: o
// columns 4c..4c+3; group 32: m, l). Thread = row, so every float4 access of a warp
// is 512 contiguous bytes.
constexpr int PARTIAL_GROUPS = D / 4 + 1;
constexpr int PARTIAL_TILE_FLOATS = PARTIAL_GROUPS * BM * 4;
static_assert(PARTIAL_TILE_FLOATS == BM * PREFILL_PARTIAL_ROW_FLOATS, "partial tile size");
constexpr int TMEM_COLS = 512;

constexpr int OFF_QA = 0;
constexpr int OFF_QB = OFF_QA + TILE;
constexpr int OFF_K = OFF_QB + TILE;
constexpr int OFF_V = OFF_K + NK * TILE;
constexpr int OFF_KMETA = OFF_V + NV * TILE;
constexpr int OFF_VMETA = OFF_KMETA + NK * BLOCKS * (int)sizeof(KMeta);
constexpr int OFF_BAR = OFF_VMETA + NV * BLOCKS * (int)sizeof(VMeta);
constexpr int NBARS = 3 + 3 * NK + 3 * NV + 7 + 2 + 2;
// float2 [2][8][64]: per segment parity, angles of rows 16 k of both Q tiles (the
// segment's base angle already added); then float2 [64][24]: angles of row offsets.
constexpr int OFF_QCS = (OFF_BAR + NBARS * 8 + 15) & ~15;
constexpr int OFF_ROWS = OFF_QCS + 2 * 8 * (D / 2) * 8;
constexpr int OFF_SCHED = OFF_ROWS + kAngleRows * (D / 2) * 8;
constexpr int SCHED_BYTES = 64;  // room for Sched (checked below)
// Mixed launches: per decode unit, whether each member passed its checks; a ring of
// 4 segments (written in the Q prologue one segment ahead, read in the deferred epilogue).
constexpr int OFF_DECOK = OFF_SCHED + SCHED_BYTES;
constexpr int DECOK_BYTES = 4 * 16 * 4;
constexpr int OFF_TMEM = OFF_DECOK + DECOK_BYTES;
constexpr int SMEM = 1024 + OFF_TMEM + 16;
static_assert(OFF_QCS % 16 == 0 && OFF_ROWS % 16 == 0, "angle rows are written as 16-byte vectors");
static_assert(SMEM <= 227 * 1024, "prefill (stream) shared memory");

// One unit's geometry. n = K tiles it needs (0: the tile holds no query row).
struct UnitDesc {
  int s, tile, hp, q0, C, row0, seq_len, nb, b_chunk, n;
  int dec;  // decode work unit (item * Hkv + KV head) in a mixed launch, else -1
};

__device__ __forceinline__ UnitDesc unit_desc(const PrefillArgs& a, int u, int P) {
  UnitDesc d;
  d.dec = -1;
  const int TP = a.T * P;
  d.s = u / TP;
  const int rem = u - d.s * TP;
  d.tile = rem / P;
  d.hp = rem - d.tile * P;
  d.q0 = __ldg(&a.cu_seqlens_q[d.s]);
  d.C = __ldg(&a.cu_seqlens_q[d.s + 1]) - d.q0;
  d.row0 = d.tile * BM;
  d.seq_len = d.nb = d.b_chunk = d.n = 0;
  if (d.C <= 0 || d.row0 >= d.C) return d;
  int seq_len = __ldg(&a.seq_lens[d.s]);
  if (seq_len < 0 || seq_len > kBlock * a.max_blocks) {
    raise_status(a.status, LAZY_DEV_BAD_LEN);
    seq_len = seq_len < 0 ? 0 : kBlock * a.max_blocks;
  }
  d.seq_len = seq_len;
  d.nb = (seq_len + kBlock - 1) / kBlock;
  d.b_chunk = max(0, d.nb - (d.C + kBlock - 1) / kBlock);  // the chunk's own keys are the last segment
  const int i_last = min(d.C, d.row0 + BM) - 1;
  const int last_block = min(d.nb - 1, d.b_chunk + i_last / kBlock);
  d.n = last_block < 0 ? 0 : last_block / BLOCKS + 1;
  return d;
}

// Decode unit ud of a mixed launch: item ud / Hkv of the shared-run plan on KV head
// ud % Hkv, one 128-row tile (members x query heads) over the item's blocks,
// n = ceil(nblk / 8) key tiles. s = the item's source sequence, nb = nblk; hp puts
// the tile on its KV head.
__device__ __forceinline__ UnitDesc dec_desc(const MixedArgs& a, int ud) {
  UnitDesc d;
  const int* rec = a.items + (size_t)(ud / a.Hkv) * LAZY_PLAN_ITEM_INTS;
  d.dec = ud;
  d.s = __ldg(&rec[0]);
  d.nb = __ldg(&rec[2]);
  const int b0 = __ldg(&rec[1]), last = __ldg(&rec[3]), nmem = __ldg(&rec[4]);
  if (d.s < 0 || d.s >= a.B_dec || b0 < 0 || d.nb < 1 || d.nb > a.max_blocks_dec - b0 || last < 1 ||
      last > kBlock || nmem < 1 || nmem * a.G > BM) {  // not a valid item: skipped
    raise_status(a.status, LAZY_DEV_LAYOUT);
    d.nb = 0;
  }
  d.hp = (ud % a.Hkv) * (a.G / 2);
  d.tile = d.q0 = d.row0 = 0;
  d.C = BM;
  d.seq_len = 0;
  d.b_chunk = INT_MAX;
  d.n = d.nb > 0 ? (d.nb + BLOCKS - 1) / BLOCKS : 0;
  return d;
}

// Rotates row i of a 128-row Q tile in place (both 64-column halves, 128-byte
// swizzled) by R_{base+i}, pre-scaled by `scale`: bq holds (cos, sin) of
// (base + 16 k) w_f at [k][f], rows the row-offset table at [f][24]. With
// row_offsets = false every row of group k takes bq[k] itself (decode units, whose
// rows are query heads of one member sequence at one rotation offset).
__device__ __forceinline__ void rotate_q_row_bq(uint8_t* sQ, int i, const float2* bq, const float2* rows,
                                                float scale, bool row_offsets = true) {
  const float2* b = bq + (i >> 4) * (D / 2);
  const int s1 = 8 + (row_offsets ? (i & 15) : 0);  // table row 0 is the identity (1, 0)
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    float2 cs[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int f = 8 * c + e;
      cs[e] = add_angles(b[f], rows[f * kAngleRows + s1]);
    }
    uint4 X = *reinterpret_cast<uint4*>(sQ + sw128(i, c));
    uint4 Y = *reinterpret_cast<uint4*>(sQ + HALF + sw128(i, c));
    rotate_chunk(X, Y, make_rot8(cs, scale));
    *reinterpret_cast<uint4*>(sQ + sw128(i, c)) = X;
    *reinterpret_cast<uint4*>(sQ + HALF + sw128(i, c)) = Y;
  }
}

// The CTA's work. Units are numbered k = 0, 1, ... over the non-empty (sequence,
// tile) groups in order, P head pairs each. When units are about equally long, the
// first D = floor(units / grid) * grid run whole, unit k on CTA k % grid (all CTAs
// start together on neighbouring units, which read the same K/V tiles at about the
// same time: L2 reuse); otherwise D = 0. The
// remaining units' K tiles are laid end to end and cut into grid ranges of W tiles:
// this CTA's range is [start, end), beginning at tile j of unit k whose first tile
// sits at position U0 of that space.
struct Sched {
  int D, start, end, k, j, U0, W;
  int e_dp, q_dp, e_sk, q_sk;  // group cursor (group, non-empty groups before it) at the first unit of each phase
};
static_assert(sizeof(Sched) <= SCHED_BYTES, "Sched must fit its shared-memory slot");
static_assert(OFF_SCHED % 16 == 0 && OFF_TMEM % 16 == 0, "shared-memory slots are 16-byte aligned");

}  // namespace

// Optional per-segment timestamps (build with -DLAZY_PREFILL_TRACE): 8 segments x 8
// u64 per CTA after the partials in the workspace: [0] first S ready (softmax), [1]
// last P V done, [2] epilogue done, [3] j0 | j1 << 16 | whole << 31, [4] Q issued
// (producer), [5] Q landed (rotation warps), [6] Q rotated, [7] first S issued (MMA).
// Segment 7 holds kernel entry [0] and the end of the scheduling prologue [1].
#ifdef LAZY_PREFILL_TRACE
#define LAZY_PF_TRACE_IF(cond, sg, i, v)                                                               \
  do {                                                                                                 \
    if ((cond) && (sg) < 8)                                                                            \
      reinterpret_cast<unsigned long long*>(a.partials + (size_t)2 * gridDim.x * 2 * PARTIAL_TILE_FLOATS) \
          [((size_t)blockIdx.x * 8 + (sg)) * 8 + (i)] = (v);                                            \
  } while (0)
// After the timestamps, 8 cycle totals per CTA over its tiles: softmax of tile A,
// row 0: [0] waiting for S and V, [1] first pass, [2] second pass and P, [3] rescale
// and hand-off, [4] tiles; MMA warp: [5] waiting for P_A and V, [6] for P_B, [7] for K.
#define LAZY_PF_COUNT(i, v)                                                                             \
  (reinterpret_cast<unsigned long long*>(a.partials + (size_t)2 * gridDim.x * 2 * PARTIAL_TILE_FLOATS) \
       [(size_t)gridDim.x * 64 + (size_t)blockIdx.x * 8 + (i)] += (v))
#define LAZY_PF_CLK(var) const long long var = clock64()
#else
#define LAZY_PF_TRACE_IF(cond, sg, i, v) \
  do {                                   \
  } while (0)
#define LAZY_PF_COUNT(i, v) \
  do {                      \
  } while (0)
#define LAZY_PF_CLK(var)
#endif
#define LAZY_PF_TRACE(sg, i, v) LAZY_PF_TRACE_IF(threadIdx.x == 0, sg, i, v)

// The decode half of a mixed launch, merged: warp w of CTA c takes (sequence s,
// query head h) pairs c * nw + w, + grid * nw, ...; out[s][h] = sum_k 2^(m_k - M) o_k /
// sum_k 2^(m_k - M) l_k over the sequence's slots k, as shared_combine_kernel. A
// sequence is merged once its decode units have all written their partials (their
// count of written rows, acquired, reaches slots x Hq); the launch is cooperative, so
// every unit is resident or done, and the wait is bounded (LAZY_DEV_TIMEOUT after it).
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void mixed_combine(const MixedArgs& a, int warp, int nw) {
  constexpr int PER = D / 32, BATCH = 8;
  const int lane = threadIdx.x & 31;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml);
  for (long long task = (long long)blockIdx.x * nw + warp; task < (long long)a.B_dec * a.Hq;
       task += (long long)gridDim.x * nw) {
    const int s = (int)(task / a.Hq), h = (int)(task - (long long)s * a.Hq);
    int k0 = __ldg(&a.slot_indptr[s]), k1 = __ldg(&a.slot_indptr[s + 1]);
    if (k0 < 0 || k1 < k0 || k1 > a.num_slots) {
      if (lane == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
      k0 = k1 = 0;
    }
    const int need = (k1 - k0) * a.Hq;  // rows: every slot holds Hq query heads
    int ok = 1;
    if (lane == 0 && need > 0) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_gpu(&a.seq_done[s]) < need) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          raise_status(a.status, LAZY_DEV_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(256);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) continue;
    float M = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    for (int kc = k0; kc < k1; kc += BATCH) {
      const int n = min(BATCH, k1 - kc);
      float2 mlj[BATCH];
      float4 vj[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        mlj[u] = make_float2(-INFINITY, 0.f);
        vj[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (u < n) {
          const size_t pidx = (size_t)(kc + u) * a.Hq + h;
          mlj[u] = __ldcg(ml + pidx);
          vj[u] = __ldcg(reinterpret_cast<const float4*>(a.ws_o + pidx * D) + lane);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < BATCH; ++u) Mn = fmaxf(Mn, mlj[u].x);
      if (Mn == -INFINITY) continue;
      const float r = ex2(M - Mn);
      L *= r;
#pragma unroll
      for (int c = 0; c < PER; ++c) acc[c] *= r;
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const float w = ex2(mlj[u].x - Mn);  // an empty slot weighs 0
        L = fmaf(w, mlj[u].y, L);
        acc[0] = fmaf(w, vj[u].x, acc[0]);
        acc[1] = fmaf(w, vj[u].y, acc[1]);
        acc[2] = fmaf(w, vj[u].z, acc[2]);
        acc[3] = fmaf(w, vj[u].w, acc[3]);
      }
      M = Mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out_dec) + ((size_t)s * a.Hq + h) * D + lane * PER;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                pack_bf16x2(acc[2] * inv, acc[3] * inv));
  }
}

template <bool LAZY, bool ALIBI = false, bool MIXED = false>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_stream_kernel(const std::conditional_t<ALIBI, PrefillAlibiArgs,
                                                   std::conditional_t<MIXED, MixedArgs, PrefillArgs>> a,
                          const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap_dec) {
  static_assert(!(ALIBI && LAZY), "the ALiBi prefill does not rotate");
  static_assert(!(ALIBI && MIXED), "mixed launches rotate");
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
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 3;
  uint64_t* k_ready = k_full + NK;
  uint64_t* k_empty = k_ready + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_ready = v_full + NV;
  uint64_t* v_empty = v_ready + NV;
  uint64_t* s_full = v_empty + NV;   // [2]: tile A, tile B
  uint64_t* p_full = s_full + 2;     // [2]
  uint64_t* pv_done = p_full + 2;    // [2]
  uint64_t* mma_drain = pv_done + 2;
  uint64_t* bcs_ready = mma_drain + 1;  // [2]: base angles of segment parity 0 / 1 written
  uint64_t* p_half = bcs_ready + 2;     // [2]: P of a tile's first 64 keys written (tile A, B)
  float2* base_cs = reinterpret_cast<float2*>(base + OFF_QCS);
  float2* angle_rows = reinterpret_cast<float2*>(base + OFF_ROWS);
  Sched* sched = reinterpret_cast<Sched*>(base + OFF_SCHED);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(base + OFF_TMEM);
  int* dec_ok = reinterpret_cast<int*>(base + OFF_DECOK);  // [4][16]
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.Hq / 2;
  const int E = a.B * a.T;  // (sequence, tile) groups; a group holds P units of equal length
  LAZY_PF_TRACE(7, 0, global_timer_ns());

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_ready, 256);
    mbar_init(q_empty, 1);
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
      mbar_init(&p_half[t], 128);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(mma_drain, 1);
    mbar_init(&bcs_ready[0], D / 2);
    mbar_init(&bcs_ready[1], D / 2);
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 12) {
    // ---------------------------------------------------------------- the CTA's work
    // Pass 1: non-empty groups (each holds P units) -> D, the units run whole.
    int ng = 0, e_dp = E, q_dp = 0, n_min = INT_MAX, n_max = 0;
    const int want_dp = blockIdx.x / P;  // non-empty group of unit blockIdx.x
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int n_e = e < E ? unit_desc(a, e * P, P).n : 0;
      n_min = min(n_min, n_e > 0 ? n_e : INT_MAX);
      n_max = max(n_max, n_e);
      const unsigned ne = __ballot_sync(0xffffffffu, n_e > 0);
      const int qe = ng + __popc(ne & ((1u << lane) - 1u));
      const unsigned hit = __ballot_sync(0xffffffffu, ((ne >> lane) & 1u) && qe == want_dp);
      if (hit && e_dp == E) {
        e_dp = e0 + __ffs(hit) - 1;
        q_dp = want_dp;
      }
      ng += __popc(ne);
    }
    const long long units = (long long)ng * P;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      n_min = min(n_min, __shfl_xor_sync(0xffffffffu, n_min, off));
      n_max = max(n_max, __shfl_xor_sync(0xffffffffu, n_max, off));
    }
    // Whole units first only when they are about equally long (otherwise whole units
    // would leave CTAs idle): max n <= 1.25 min n.
    const bool uniform = (long long)n_max * 4 <= (long long)n_min * 5;
    const int D = uniform ? (int)(units / gridDim.x * gridDim.x) : 0;
    // Pass 2: K tiles of the units k >= D, laid end to end; find this CTA's start.
    long long pos = 0, tot = 0;
    int q_before = 0, k_s = 0, j_s = 0, U0_s = 0, e_sk = E, q_sk = 0;
    bool found = false;
    long long W = 0, st = 0;
    for (int pass = 0; pass < 2; ++pass) {
      pos = 0;
      q_before = 0;
      if (pass == 1) {
        W = (tot + gridDim.x - 1) / gridDim.x;
        st = min(tot, W * blockIdx.x);
      }
      for (int e0 = 0; e0 < E && !(pass == 1 && (found || st >= tot)); e0 += 32) {
        const int e = e0 + lane;
        const int n = e < E ? unit_desc(a, e * P, P).n : 0;
        const unsigned ne = __ballot_sync(0xffffffffu, n > 0);
        const int q = q_before + __popc(ne & ((1u << lane) - 1u));  // this group's index among non-empty ones
        const int h0 = n > 0 ? min(P, max(0, D - q * P)) : P;      // first head pair of the group past D
        const long long cnt = (long long)(P - h0) * n;              // the group's tiles in the split space
        long long inc = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, inc, off);
          if (lane >= off) inc += v;
        }
        const long long excl = pos + inc - cnt;
        if (pass == 1) {
          const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && st >= excl && st < excl + cnt);
          if (hit) {
            const int l = __ffs(hit) - 1;
            const long long off = __shfl_sync(0xffffffffu, st - excl, l);
            const int nl = __shfl_sync(0xffffffffu, n, l), ql = __shfl_sync(0xffffffffu, q, l);
            const int hl = __shfl_sync(0xffffffffu, h0, l);
            const int hp = hl + (int)(off / nl);
            k_s = ql * P + hp;
            j_s = (int)(off % nl);
            e_sk = e0 + l;
            q_sk = ql;
            U0_s = (int)(__shfl_sync(0xffffffffu, excl, l) + (long long)(hp - hl) * nl);
            found = true;
          }
        }
        pos += __shfl_sync(0xffffffffu, inc, 31);
        q_before += __popc(ne);
      }
      if (pass == 0) tot = pos;
    }
    if (tot > INT_MAX || units > INT_MAX) {
      if (lane == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
      tot = 0;
    }
    const long long en = min(tot, st + W);
    if (lane == 0)
      *sched = Sched{D, found ? (int)st : 0, found ? (int)en : 0, k_s, j_s, U0_s, (int)W, e_dp, q_dp, e_sk, q_sk};
  }
  if (warp >= 8 && warp < 12) load_angle_rows(angle_rows, a.rope, threadIdx.x - 256, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const Sched sc = *sched;
  LAZY_PF_TRACE(7, 1, global_timer_ns());

  // Walks the CTA's segments: its whole units first, then its range of the split
  // space. body(u, unit, j0, j1, U0, sg, has_next, next_unit) per segment, U0 =
  // position of unit u's first tile in the split space (-1 for a whole unit), sg =
  // segment index, next_unit = the following segment's unit (for work done ahead).
  // body returns false to stop.
  auto for_segments = [&](auto&& body) {
    struct Seg {
      int u, j0, j1, U0;
      UnitDesc un;
    };
    // Cursor over the groups: e, its description, and q = non-empty groups before e;
    // it starts at the first unit of the CTA's first phase and jumps to the split
    // phase's first unit (both found by the range scan).
    const bool dp = (int)blockIdx.x < sc.D;
    int e = dp ? sc.e_dp : sc.e_sk, q = dp ? sc.q_dp : sc.q_sk;
    UnitDesc gd = unit_desc(a, (e < E ? e : 0) * P, P);
    bool in_sk = !dp;
    auto seek = [&](int k) {  // move to the non-empty group holding unit k
      const int want = k / P;
      while (e < E && !(gd.n > 0 && q == want)) {
        if (gd.n > 0) ++q;
        ++e;
        if (e < E) gd = unit_desc(a, e * P, P);
      }
    };
    int kd = blockIdx.x;                                     // next whole unit
    int x = sc.start, ks = sc.k, jn = sc.j, U0n = sc.U0;     // split-space cursor
    int kdec = blockIdx.x;                                   // next decode unit (mixed launches)
    (void)kdec;
    auto next = [&](Seg& sgm) -> bool {
      if constexpr (MIXED) {  // decode units first, whole, dealt round robin
        while (kdec < a.num_items * a.Hkv) {
          sgm.un = dec_desc(a, kdec);
          kdec += gridDim.x;
          if (sgm.un.n == 0) continue;  // an invalid item (flagged)
          sgm.u = -1;
          sgm.j0 = 0;
          sgm.j1 = sgm.un.n;
          sgm.U0 = -1;
          return true;
        }
      }
      if (kd < sc.D) {
        seek(kd);
        sgm.un = gd;
        sgm.un.hp = kd - (kd / P) * P;
        sgm.u = e * P + sgm.un.hp;
        sgm.j0 = 0;
        sgm.j1 = gd.n;
        sgm.U0 = -1;
        kd += gridDim.x;
        return true;
      }
      if (x < sc.end) {
        if (!in_sk) {  // jump to the split phase's first group
          in_sk = true;
          if (sc.e_sk > e) {
            e = sc.e_sk;
            q = sc.q_sk;
            gd = unit_desc(a, e * P, P);
          }
        }
        seek(ks);
        sgm.un = gd;
        sgm.un.hp = ks - (ks / P) * P;
        sgm.u = e * P + sgm.un.hp;
        sgm.j0 = jn;
        sgm.j1 = min(gd.n, jn + (sc.end - x));
        sgm.U0 = U0n;
        x += sgm.j1 - jn;
        U0n += gd.n;
        ++ks;
        jn = 0;
        return true;
      }
      return false;
    };
    Seg cur, nxt;
    bool have = next(cur);
    for (int sg = 0; have; ++sg) {
      const bool have_nxt = next(nxt);
      if (!body(cur.u, cur.un, cur.j0, cur.j1, cur.U0, sg, have_nxt, nxt.un)) return;
      cur = nxt;
      have = have_nxt;
    }
  };

  if (warp == 12 || warp == 14) {
    // ---------------------------------------------------------------- TMA producers
    const bool is_v = warp == 14;
    if (lane == 0) tma_prefetch_map(is_v ? &vmap : &kmap);
    if (!is_v && lane == 0) tma_prefetch_map(&qmap);
    const int ns = is_v ? NV : NK;
    uint64_t* ful_ring = is_v ? v_full : k_full;
    uint64_t* emp_ring = is_v ? v_empty : k_empty;
    uint8_t* ring = is_v ? sV : sK;
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    int g = 0, qs = 0;  // tiles issued, Q loads issued
    bool ok = true;
    for_segments([&](int u, const UnitDesc& un, int j0, int j1, int U0, int sg, bool, const UnitDesc&) {
      (void)u;
      (void)U0;
      const int kvh = (2 * un.hp) / a.G;
      const bool dec = MIXED && un.dec >= 0;
      if (!is_v) {  // Q of both tiles; the previous segment's S products must be done with sQ
        if (sg > 0 && !warp_wait(q_empty, (sg - 1) & 1, a.status)) return ok = false;
        LAZY_PF_TRACE_IF(lane == 0, sg, 4, global_timer_ns());
        if (dec) {
          if constexpr (MIXED) {
            // Decode unit: tile A's row r = member (r / G) x query head (r % G) of this KV
            // head; tile B idles through the unit.
            const int* rec = a.items + (size_t)(un.dec / a.Hkv) * LAZY_PLAN_ITEM_INTS;
            const int nmem = min(__ldg(&rec[4]), BM / a.G);
            if (lane == 0) {
              mbar_arrive_expect_tx(q_full, (uint32_t)nmem * (uint32_t)a.G * 256u);
              for (int m = 0; m < nmem; ++m) {
                const int seq = min(max(__ldg(&rec[8 + 4 * m]), 0), a.B_dec - 1);
                tma_load_3d(sQ[0] + m * a.G * 128, &qmap_dec, q_full, 0, kvh * a.G, seq);
                tma_load_3d(sQ[0] + HALF + m * a.G * 128, &qmap_dec, q_full, 64, kvh * a.G, seq);
              }
            }
          }
        } else if (lane == 0) {
          mbar_arrive_expect_tx(q_full, 2 * TILE);
          for (int t = 0; t < 2; ++t) {
            tma_load_3d(sQ[t], &qmap, q_full, 0, 2 * un.hp + t, un.q0 + un.row0);
            tma_load_3d(sQ[t] + HALF, &qmap, q_full, 64, 2 * un.hp + t, un.q0 + un.row0);
          }
        }
        qs = sg + 1;
      }
      // (decode units read the decode batch's words, below; nb_pf = 0 keeps them away
      // from the prefill words)
      const int nb_pf = dec ? 0 : un.nb;
      const uint32_t* wrow = a.words + (size_t)(dec ? 0 : un.s) * a.max_blocks;
      // Block words 32 at a time, a chunk ahead: lane l holds block cbase + l (wcur) and
      // cbase + 32 + l (wnext).
      int cbase = (j0 * BLOCKS) & ~31;
      uint32_t wcur = cbase + lane < nb_pf ? __ldg(&wrow[cbase + lane]) : 0u;
      uint32_t wnext = cbase + 32 + lane < nb_pf ? __ldg(&wrow[cbase + 32 + lane]) : 0u;
      for (int j = j0; j < j1; ++j, ++g) {
        // ALiBi walks a unit's tiles from the last (the keys nearest the queries, with
        // the largest bias) to the first, so that the running maximum is met early and
        // later tiles seldom raise it (each raise rescales the running output).
        const int jt = ALIBI ? j0 + j1 - 1 - j : j;
        uint32_t w;
        const int b = jt * BLOCKS + min(lane, BLOCKS);
        if constexpr (ALIBI) {
          w = (lane <= BLOCKS && b < nb_pf) ? __ldg(&wrow[b]) : 0u;
        } else {
          if (j * BLOCKS >= cbase + 32) {  // warp-uniform: the tile starts in the next chunk
            cbase += 32;
            wcur = wnext;
            wnext = cbase + 32 + lane < nb_pf ? __ldg(&wrow[cbase + 32 + lane]) : 0u;
          }
          // Lanes 0..BLOCKS-1 describe the tile's blocks; lane BLOCKS takes the next block's
          // word so that the tile's last block knows where the following one starts.
          const int rel = b - cbase;  // 0 .. 40
          const uint32_t w0 = __shfl_sync(0xffffffffu, wcur, rel & 31);
          const uint32_t w1 = __shfl_sync(0xffffffffu, wnext, rel & 31);
          w = (lane <= BLOCKS && b < nb_pf) ? (rel < 32 ? w0 : w1) : 0u;
        }
        BlockInfo bi = decode_word(w, b, a.id_bits);
        const int p_after = __shfl_down_sync(0xffffffffu, bi.p, 1);
        int y = -kBlock, nv = 0;  // rows of an invalid block start at -16: read as zeros
        if constexpr (MIXED) {
          if (dec) {  // item block b of the source sequence's run: full but the last
            const int* rec = a.items + (size_t)(un.dec / a.Hkv) * LAZY_PLAN_ITEM_INTS;
            const uint32_t wd = (lane < BLOCKS && b < un.nb)
                                    ? __ldg(&a.words_dec[(size_t)un.s * a.max_blocks_dec + __ldg(&rec[1]) + b])
                                    : 0u;
            bi.phys = (int)(wd & ((1u << a.id_bits) - 1u));
            bi.p = 0;
          }
        }
        if (lane < BLOCKS && b < un.nb) {
          bool item_nv = false;
          if constexpr (MIXED) {
            if (dec) {
              const int* rec = a.items + (size_t)(un.dec / a.Hkv) * LAZY_PLAN_ITEM_INTS;
              nv = b == un.nb - 1 ? min(max(__ldg(&rec[3]), 0), kBlock) : kBlock;
              item_nv = true;
            }
          }
          if (!item_nv) {
            nv = block_valid(b, un.nb, un.seq_len, bi.p, b + 1 < un.nb ? p_after : bi.p);
            nv = nv < 0 ? 0 : (nv > kBlock ? kBlock : nv);
          }
          if (bi.phys < a.num_pool_blocks) {
            y = (bi.phys * a.Hkv + kvh) * kBlock;
          } else {
            if (!is_v) raise_status(a.status, LAZY_DEV_BAD_BLOCK_ID);
            nv = 0;
          }
        }
        const int ybox = __shfl_sync(0xffffffffu, y, (lane >> 1) & 7);  // lane l loads half l & 1 of block l >> 1
        const int st = g % ns;
        if (g >= ns && !warp_wait(&emp_ring[st], ((g / ns) & 1) ^ 1, a.status)) return ok = false;
        if (lane < BLOCKS) {
          if (is_v)
            vmeta[st * BLOCKS + lane] = VMeta{nv, b >= un.b_chunk ? kBlock * (b - un.b_chunk) : -1, bi.p, 0};
          else
            kmeta[st * BLOCKS + lane] = KMeta{bi.p, nv};
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&ful_ring[st], TILE);
        __syncwarp();
        if (lane < 2 * BLOCKS)
          tma_load_2d(ring + st * TILE + (lane & 1) * HALF + (lane >> 1) * (kBlock * 128), map, &ful_ring[st],
                      (lane & 1) * 64, ybox);
      }
      return true;
    });
    if (!ok) abort_flag = 1;
    LAZY_PF_TRACE_IF(lane == 0, 7, is_v ? 5 : 4, global_timer_ns());
    if (lane == 0) {  // every copy issued must land before the CTA exits (bounded)
      if (!is_v && qs > 0) mbar_wait(q_full, (qs - 1) & 1, a.status);
      for (int j = max(0, g - ns); j < g; ++j) mbar_wait(&ful_ring[j % ns], (j / ns) & 1, a.status);
    }
  } else if (warp == 13) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idO = idesc_bf16_f32(BM, D, true);
      // Descriptors are built once; a byte offset moves the 14-bit start-address
      // field by offset >> 4 (shared addresses stay below 2^18, so it never carries).
      const uint64_t dQ[2] = {sdesc_sw128(smem_u32(sQ[0]), 16, 1024), sdesc_sw128(smem_u32(sQ[1]), 16, 1024)};
      const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(sV), HALF, 1024);
      auto issue_s = [&](int g, int t) {
        const uint64_t k0 = dK + (uint64_t)(((g % NK) * TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = ((ks >> 2) * HALF + (ks & 3) * 32) >> 4;
          tc_mma(tmem + 128 * t, dQ[t] + off, k0 + off, idS, ks > 0);
        }
        tc_commit(&s_full[t]);
      };
      // P V over the 64 keys from 16 ks0 (P_t: 8 TMEM columns, 16 keys, per k-step); the
      // second half commits pv_done.
      auto issue_pv = [&](int g, int t, bool acc, int ks0) {
        const uint64_t v0 = dV + (uint64_t)(((g % NV) * TILE) >> 4);
#pragma unroll
        for (int k = 0; k < BN / 32; ++k) {
          const int ks = ks0 + k;
          tc_mma_ta(tmem + 256 + 128 * t, tmem + 128 * t + 8 * ks, v0 + (uint32_t)(ks * 2048 >> 4), idO,
                    (acc || ks > 0) ? 1u : 0u);
        }
        if (ks0 > 0) tc_commit(&pv_done[t]);
      };
      int g = 0;   // tiles whose S has been issued == tiles started
      int gb = 0;  // tiles tile B has taken part in (it idles through decode units)
      bool ok = true;
      for_segments([&](int u, const UnitDesc& un, int j0, int j1, int U0, int sg, bool, const UnitDesc&) {
        (void)u;
        (void)U0;
        const bool two = !(MIXED && un.dec >= 0);  // both tiles (prefill) or tile A only (decode)
        // The segment's first S pair: its Q is rotated. S_t overwrites P_t of the previous
        // tile, whose P V was issued earlier by this thread: one thread's MMAs execute in
        // issue order, so that P V has read P_t before S_t writes the columns.
        ok = mbar_wait(q_ready, sg & 1, a.status) && mbar_wait(&k_ready[g % NK], (g / NK) & 1, a.status);
        if (!ok) return false;
        tc_fence_after();
        issue_s(g, 0);
        if (two) issue_s(g, 1);
        LAZY_PF_TRACE_IF(true, sg, 7, global_timer_ns());
        tc_commit(&k_empty[g % NK]);
        if (j1 - j0 == 1) tc_commit(q_empty);  // the segment's last S product is issued
        for (int j = j0; j < j1; ++j, ++g) {
          const bool more = j + 1 < j1;
          // V(g) before P_A(g): each wait on a shared-memory barrier takes a round trip
          // that the tensor core's operand reads make long, and V(g) is usually ready
          // first. (v_ready is arrived only after V(g) has landed, so it covers v_full.)
          // P V of each tile in two halves: the first 64 keys' P is handed over while the
          // softmax still computes the rest, so its products run meanwhile.
          LAZY_PF_CLK(c0);
          ok = mbar_wait(&v_ready[g % NV], (g / NV) & 1, a.status) && mbar_wait(&p_half[0], g & 1, a.status);
          if (!ok) return false;
          tc_fence_after();
          issue_pv(g, 0, j > j0, 0);
          ok = mbar_wait(&p_full[0], g & 1, a.status);
          LAZY_PF_CLK(c1);
          LAZY_PF_COUNT(5, c1 - c0);
          if (!ok) return false;
          tc_fence_after();
          issue_pv(g, 0, j > j0, BN / 32);
          if (more) {  // S_A(g+1) overwrites P_A(g), read by PV_A(g) issued just above (in order)
            LAZY_PF_CLK(c2);
            ok = mbar_wait(&k_ready[(g + 1) % NK], ((g + 1) / NK) & 1, a.status);
            LAZY_PF_CLK(c3);
            LAZY_PF_COUNT(7, c3 - c2);
            if (!ok) return false;
            tc_fence_after();
            issue_s(g + 1, 0);
          }
          if (two) {
            LAZY_PF_CLK(c4);
            ok = mbar_wait(&p_half[1], gb & 1, a.status);
            if (!ok) return false;
            tc_fence_after();
            issue_pv(g, 1, j > j0, 0);
            ok = mbar_wait(&p_full[1], gb & 1, a.status);
            LAZY_PF_CLK(c5);
            LAZY_PF_COUNT(6, c5 - c4);
            if (!ok) return false;
            tc_fence_after();
            issue_pv(g, 1, j > j0, BN / 32);
          }
          tc_commit(&v_empty[g % NV]);
          if (more) {
            if (two) issue_s(g + 1, 1);
            tc_commit(&k_empty[(g + 1) % NK]);
            if (j + 2 == j1) tc_commit(q_empty);  // the segment's last S product is issued
          }
          if (two) ++gb;
        }
        return true;
      });
      if (!ok) abort_flag = 1;
      LAZY_PF_TRACE_IF(true, 7, 3, global_timer_ns());
      tc_commit(mma_drain);
      mbar_wait(mma_drain, 0, a.status);
    }
    __syncwarp();
  } else if (warp >= 8 && warp < 12) {
    // ---------------------------------------------------------------- Q prologue, K rotation, V holes
    const int r = threadIdx.x - 256;  // 0..127
    const int c = r & 7, rb = r >> 3;  // 16-byte chunk (8 frequencies) and row within a block
    Rot8 rot;
    int p_cached = INT_MIN;
    int g = 0;
    bool ok = true;
    for_segments([&](int u, const UnitDesc& un, int j0, int j1, int U0, int sg, bool, const UnitDesc&) {
      (void)u;
      (void)U0;
      (void)un;
      (void)sg;
      for (int j = j0; j < j1; ++j, ++g) {
        const int st = g % NK;
        if (!warp_wait(&k_full[st], (g / NK) & 1, a.status)) return ok = false;
        uint8_t* kt = sK + st * TILE;
        // The tile's block records and its data are read up front, four blocks' chunks
        // per round: shared-memory loads wait long behind the tensor core's operand
        // reads, so they are issued together rather than one block at a time.
        KMeta km[BLOCKS];
        bool holes = false;
#pragma unroll
        for (int bl = 0; bl < BLOCKS; ++bl) {
          km[bl] = kmeta[st * BLOCKS + bl];
          holes |= km[bl].nvalid < kBlock;
        }
        if constexpr (LAZY) {
          if (!(MIXED && un.dec >= 0)) {  // decode units: K as stored
#pragma unroll 1
            for (int h = 0; h < BLOCKS; h += 4) {
              uint4 X[4], Y[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t off = (h + u) * (kBlock * 128) + sw128(rb, c);
                X[u] = *reinterpret_cast<const uint4*>(kt + off);
                Y[u] = *reinterpret_cast<const uint4*>(kt + HALF + off);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const KMeta m = h == 0 ? km[u] : km[4 + u];
                if (m.nvalid > 0) {
                  if (m.p != p_cached) {
                    rot = block_rot8(a.rope, c, m.p, a.status);
                    p_cached = m.p;
                  }
                  rotate_chunk(X[u], Y[u], rot);
                  const uint32_t off = (h + u) * (kBlock * 128) + sw128(rb, c);
                  *reinterpret_cast<uint4*>(kt + off) = X[u];
                  *reinterpret_cast<uint4*>(kt + HALF + off) = Y[u];
                }
              }
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&k_ready[st]);
        // v_ready(g) is arrived only after V(g) has landed, so no v_ready phase can run
        // two tiles ahead of the MMA warp (V(g+2) needs the P V products of tile g first).
        const int vs = g % NV;
        if (!warp_wait(&v_full[vs], (g / NV) & 1, a.status)) return ok = false;
        if (__any_sync(0xffffffffu, holes)) {  // hole slots' V rows may hold anything: zero them
          uint8_t* vt = sV + vs * TILE;
#pragma unroll 1
          for (int bl = 0; bl < BLOCKS; ++bl) {
            if (rb >= vmeta[vs * BLOCKS + bl].nvalid) {
              const uint32_t off = bl * (kBlock * 128) + sw128(rb, c);
              *reinterpret_cast<uint4*>(vt + off) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vt + HALF + off) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(&v_ready[vs]);
      }
      return true;
    });
    if (!ok) abort_flag = 1;
    LAZY_PF_TRACE_IF(r == 0, 7, 6, global_timer_ns());
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax, tile t
    const int t = warp >> 2;
    const int i = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + 128 * t, tO = tmem + 256 + 128 * t;
    // g counts every tile (the K/V rings' phases); gt the tiles this query tile took part
    // in (its own barriers' phases; tile B idles through decode units of a mixed launch)
    int g = 0, gt = 0;
    bool ok = true;
    // Angles of the 8 row multiples of 16 of segment sg's tiles (its base angle added),
    // into buffer sg & 1. Computed one segment ahead; rewriting a buffer for segment
    // sg + 2 happens after this thread passed q_full(sg + 1), which needs every
    // thread's q_ready(sg), i.e. its last read of the buffer for segment sg.
    auto make_bq = [&](const UnitDesc& un, int sg) {
      if (threadIdx.x < D / 2) {
        float2* bq = base_cs + (sg & 1) * 8 * (D / 2);
        const int f = threadIdx.x;
        if (MIXED && un.dec >= 0) {
          if constexpr (MIXED) {
            // Decode unit: rows of member m (16-row groups k with 16 k / G == m) are rotated
            // by R_{m_pos - p}, p = the member's document start from its own first block
            // word, whose block must be the item's (else the member is dropped).
            const int* rec = a.items + (size_t)(un.dec / a.Hkv) * LAZY_PLAN_ITEM_INTS;
            const int nmem = min(__ldg(&rec[4]), BM / a.G), b0 = __ldg(&rec[1]);
            const uint32_t id_mask = (1u << a.id_bits) - 1u;
            const uint32_t src_phys = __ldg(&a.words_dec[(size_t)un.s * a.max_blocks_dec + b0]) & id_mask;
            const float2 tf = __ldg(&a.rope[f]);
            int m_prev = -1;
            float2 cs = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int k = 0; k < 8; ++k) {
              const int m = (16 * k) / a.G;
              if (m != m_prev) {
                m_prev = m;
                bool good = false;
                if (m < nmem) {
                  const int seq = __ldg(&rec[8 + 4 * m]), bm = __ldg(&rec[8 + 4 * m + 1]);
                  const int slot = __ldg(&rec[8 + 4 * m + 2]);
                  good = seq >= 0 && seq < a.B_dec && bm >= 0 && bm <= a.max_blocks_dec - un.nb && slot >= 0 &&
                         slot < a.num_slots;
                  if (good) {
                    const BlockInfo mi = decode_word(__ldg(&a.words_dec[(size_t)seq * a.max_blocks_dec + bm]), bm,
                                                     a.id_bits);
                    good = (uint32_t)mi.phys == src_phys;
                    if (good) cs = rope_cs(tf, __ldg(&a.q_pos[seq]) - mi.p, a.status);
                  }
                  if (!good && f == 0) raise_status(a.status, LAZY_DEV_LAYOUT);
                  if (f == 0) dec_ok[(sg & 3) * 16 + m] = good;
                }
                if (!good) cs = make_float2(0.f, 0.f);  // a dropped member's rows are 0
              }
              bq[k * (D / 2) + f] = cs;
            }
          }
        } else {
          const float2 b = rope_cs(__ldg(&a.rope[f]), __ldg(&a.q_start[un.s]) + un.row0, a.status);
#pragma unroll
          for (int k = 0; k < 8; ++k) bq[k * (D / 2) + f] = add_angles(b, angle_rows[f * kAngleRows + k]);
        }
        mbar_arrive(&bcs_ready[sg & 1]);
      }
    };
    // The finished segment whose epilogue still has to run (it runs after the next
    // segment's Q prologue, so that the tensor core starts the next segment sooner).
    struct Pend {
      UnitDesc un;
      int j0, j1, U0, g_last, sg;
      float m_run, l_run;
      bool valid;
    } pend;
    pend.valid = false;
    // ---- epilogue of a finished segment: O / l -> bf16 for a whole unit; for a piece of a
    // unit cut by range boundaries, this row's fp32 partial goes to the CTA's slot (2c for
    // its first segment, 2c+1 for its last), and the thread that completes the row's
    // arrival count merges the pieces.
    auto epilogue = [&](const Pend& pd) -> bool {
      if constexpr (MIXED) {
        if (pd.un.dec >= 0) {
          // Decode unit: tile A's rows (member m = row / G, query head row % G of the
          // KV head) go to the members' partial slots; tile B repeated them.
          if (t == 1) return true;
          if (!warp_wait(&pv_done[0], pd.g_last & 1, a.status)) return false;
          tc_fence_after();
          const int* rec = a.items + (size_t)(pd.un.dec / a.Hkv) * LAZY_PLAN_ITEM_INTS;
          const int nmem = min(__ldg(&rec[4]), BM / a.G), kvh = (2 * pd.un.hp) / a.G;
          const int m = i / a.G, h = i - m * a.G;
          const int slot = m < nmem ? __ldg(&rec[8 + 4 * m + 2]) : -1;
          const bool slot_ok = slot >= 0 && slot < a.num_slots;
          // a member that failed its checks leaves an empty partial (weight 0 in the merge)
          const bool good = slot_ok && dec_ok[(pd.sg & 3) * 16 + m];
          const size_t pidx = ((size_t)(slot_ok ? slot : 0) * a.Hq + (size_t)kvh * a.G + h);
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            float o[32];
            tmem_ld32(tO + lane_base + 32 * q, o);
            tmem_ld_wait(o);
            if (slot_ok) {
              float4* dst = reinterpret_cast<float4*>(a.ws_o + pidx * D + 32 * q);
#pragma unroll
              for (int k = 0; k < 32; k += 4)
                dst[k / 4] = good ? make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          if (slot_ok)
            *reinterpret_cast<float2*>(a.ws_ml + 2 * pidx) =
                good ? make_float2(pd.m_run, pd.l_run) : make_float2(-INFINITY, 0.f);
          // Count this row as written for its sequence (the merge waits for slots x Hq
          // rows): each thread fences its own writes, then one lane per sequence in the
          // warp adds its lanes' rows. No barrier beyond the warp: a warp whose wait gave
          // up never holds the others.
          __threadfence();
          __syncwarp();
          const int seq = slot_ok ? __ldg(&rec[8 + 4 * m]) : -1;
          const bool counts = seq >= 0 && seq < a.B_dec;
          const unsigned same = __match_any_sync(0xffffffffu, counts ? seq : -1);
          if (counts && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&a.seq_done[seq], __popc(same));
          return true;
        }
      }
      if (!warp_wait(&pv_done[t], pd.g_last & 1, a.status)) return false;
      LAZY_PF_TRACE(pd.sg, 1, global_timer_ns());
      LAZY_PF_TRACE(pd.sg, 3, (unsigned long long)pd.j0 | ((unsigned long long)pd.j1 << 16) |
                                  ((unsigned long long)(pd.j0 == 0 && pd.j1 == pd.un.n) << 31));
      tc_fence_after();
      const UnitDesc& un = pd.un;
      const int iq = un.row0 + i;
      const int h = 2 * un.hp + t;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(un.q0 + iq) * a.Hq + h) * D;
      const bool row_live = iq < un.C;
      auto store_row = [&](const float (&o)[32], int q, float inv) {
        if (row_live) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 v = make_uint4(pack_bf16x2(o[k] * inv, o[k + 1] * inv), pack_bf16x2(o[k + 2] * inv, o[k + 3] * inv),
                                 pack_bf16x2(o[k + 4] * inv, o[k + 5] * inv), pack_bf16x2(o[k + 6] * inv, o[k + 7] * inv));
            *reinterpret_cast<uint4*>(dst + 32 * q + k) = v;
          }
        }
      };
      if (pd.j0 == 0 && pd.j1 == un.n) {  // whole unit
        const float inv = pd.l_run > 0.f ? 1.f / pd.l_run : 0.f;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(tO + lane_base + 32 * q, o);
          tmem_ld_wait(o);
          store_row(o, q, inv);
        }
        LAZY_PF_TRACE(pd.sg, 2, global_timer_ns());
        return true;
      }
      const int c0 = pd.U0 / sc.W, c1 = (pd.U0 + un.n - 1) / sc.W;  // CTAs holding pieces of u
      const int npieces = c1 - c0 + 1;
      auto slot_of = [&](int cc) { return (cc * sc.W >= pd.U0) ? 2 * cc : 2 * cc + 1; };
      // float4 column group cg of this row in a slot: base + cg * BM
      auto piece = [&](int cc) {
        return reinterpret_cast<float4*>(a.partials + ((size_t)slot_of(cc) * 2 + t) * PARTIAL_TILE_FLOATS) + i;
      };
      float4* ptile = piece(blockIdx.x);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float o[32];
        tmem_ld32(tO + lane_base + 32 * q, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int k = 0; k < 32; k += 4) ptile[(8 * q + k / 4) * BM] = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
      }
      ptile[(D / 4) * BM] = make_float4(pd.m_run, pd.l_run, 0.f, 0.f);
      __threadfence();
      // The counter of the split belongs to the first range boundary inside the unit.
      int* cnt = a.counters + ((size_t)(c0 + 1) * 2 + t) * BM + i;
      const int arrived = atomicAdd(cnt, 1) + 1;
      LAZY_PF_TRACE(pd.sg, 2, global_timer_ns());
      if (arrived != npieces) return true;
      __threadfence();
      // (m, l) of every piece, then the weights 2^(m_p - M): up to 8 pieces in registers.
      float M = -INFINITY, L = 0.f;
      float mp[8], lp[8];
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const float4 ml = pc < npieces ? __ldcg(piece(c0 + pc) + (D / 4) * BM) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        mp[pc] = ml.x, lp[pc] = ml.y;
      }
      for (int pc = 8; pc < npieces; ++pc) M = fmaxf(M, __ldcg(piece(c0 + pc) + (D / 4) * BM).x);
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) M = fmaxf(M, mp[pc]);
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) L += (M == -INFINITY ? 0.f : ex2(mp[pc] - M)) * lp[pc];
      for (int pc = 8; pc < npieces; ++pc) {
        const float4 ml = __ldcg(piece(c0 + pc) + (D / 4) * BM);
        L += (M == -INFINITY ? 0.f : ex2(ml.x - M)) * ml.y;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float o[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0.f;
        for (int pc = 0; pc < npieces; ++pc) {
          const float4* pr = piece(c0 + pc);
          const float w = M == -INFINITY ? 0.f : ex2((pc < 8 ? mp[pc] : __ldcg(pr + (D / 4) * BM).x) - M);
          float4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] = __ldcg(pr + (8 * q + k) * BM);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            o[4 * k] += w * v[k].x, o[4 * k + 1] += w * v[k].y, o[4 * k + 2] += w * v[k].z, o[4 * k + 3] += w * v[k].w;
          }
        }
        store_row(o, q, inv);
      }
      return true;
    };
    // A K tile's masks for this row: the valid keys of each of its blocks (8 bits per
    // block; holes, and the causal limit inside the chunk), whether all its keys are
    // valid for every row, and (ALiBi) each block's bias slope (n0 - m_i) in log2 units.
    struct TileMask {
      uint64_t lim;
      bool full;
      float b0[ALIBI ? BLOCKS : 1];
    };
    auto read_mask = [&](int vs, int iq, float slope2, int m_row) {
      TileMask tm;
      tm.lim = 0;
      tm.full = true;
#pragma unroll
      for (int bl = 0; bl < BLOCKS; ++bl) {
        const VMeta m = vmeta[vs * BLOCKS + bl];
        tm.full &= (m.nvalid == kBlock) & (m.chunk_j0 < 0);
        const int l = m.chunk_j0 >= 0 ? max(0, min(m.nvalid, iq - m.chunk_j0 + 1)) : m.nvalid;
        tm.lim |= (uint64_t)(uint32_t)l << (8 * bl);
        if constexpr (ALIBI) tm.b0[bl] = slope2 * (float)(m.pos - m_row);
      }
      return tm;
    };
    for_segments([&](int u, const UnitDesc& un, int j0, int j1, int U0, int sg, bool has_next,
                     const UnitDesc& next_un) {
      (void)u;
      const int iq = un.row0 + i;  // query index within the chunk
      // ALiBi: slope of this tile's query head in log2 units and the row's position m_i.
      float slope2 = 0.f;
      int m_row = 0;
      if constexpr (ALIBI) {
        slope2 = __ldg(&a.alibi[2 * un.hp + t]) * 1.4426950408889634f;
        m_row = __ldg(&a.q_start[un.s]) + iq;
      }
      // Q prologue: R_{m_i} of row i of tile t, m_i = q_start + row0 + i, pre-scaled by
      // sm_scale * log2(e).
      if (sg == 0) make_bq(un, 0);
      ok = warp_wait(&bcs_ready[sg & 1], (sg >> 1) & 1, a.status) && warp_wait(q_full, sg & 1, a.status);
      if (!ok) return false;
      LAZY_PF_TRACE(sg, 5, global_timer_ns());
      // Tile B idles through a decode unit (its Q buffer is not loaded), but still
      // counts in the segment's Q handshake.
      const bool idle = MIXED && un.dec >= 0 && t == 1;
      if (!idle)
        rotate_q_row_bq(sQ[t], i, base_cs + (sg & 1) * 8 * (D / 2), angle_rows, a.scale_log2,
                        !(MIXED && un.dec >= 0));
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
      LAZY_PF_TRACE(sg, 6, global_timer_ns());
      if (has_next) make_bq(next_un, sg + 1);
      if (pend.valid) {
        ok = epilogue(pend);
        pend.valid = false;
        if (!ok) return false;
      }
      if (idle) {
        g += j1 - j0;
        return true;
      }
      float m_run = -INFINITY, l_run = 0.f;
      // The key limits of a tile are read from its V metadata one tile ahead, while the
      // tensor core still computes its S: shared-memory loads wait long behind the
      // products' operand reads, and this keeps them off the softmax's path.
      if (!warp_wait(&v_full[g % NV], (g / NV) & 1, a.status)) return ok = false;
      TileMask tm = read_mask(g % NV, iq, slope2, m_row);
      for (int j = j0; j < j1; ++j, ++g, ++gt) {
        LAZY_PF_CLK(k0);
        ok = warp_wait(&s_full[t], gt & 1, a.status);
        LAZY_PF_CLK(k1);
        if (!ok) return false;
        if (j == j0) LAZY_PF_TRACE(sg, 0, global_timer_ns());
        tc_fence_after();
        const bool full_tile = tm.full;
        // Valid keys of block b for this row (holes; causal inside the chunk).
        auto limb = [&](int b) { return (int)((tm.lim >> (8 * b)) & 0xffu); };
        // ALiBi bias of key k (0..31) of chunk q (blocks 2q, 2q + 1): slope (n - m_i) =
        // b0 + slope (k & 15), with b0 = slope (n0 - m_i) of the key's block.
        auto bias0 = [&](int q, int h2) {
          const int b = 2 * q + h2;
          float r = tm.b0[0];
#pragma unroll
          for (int e = 1; e < BLOCKS; ++e) r = b == e ? tm.b0[e] : r;
          return r;
        };
        // Maximum of chunk q (keys 32 q .. 32 q + 31) over the row's valid keys. ALiBi: an
        // upper bound of the biased maximum, each block's largest score plus the largest
        // bias in the block, b0 + max(0, 15 slope). It exceeds the exact maximum by at
        // most 15 |slope| (log2 units), so the second pass's weights shrink by at most
        // that factor, far inside fp32 and bf16 range; the softmax itself is unchanged.
        auto chunk_max = [&](const float(&sv)[32], int q) {
          if constexpr (ALIBI) {
            const float kmax = fmaxf(0.f, 15.f * slope2);
            float mx = -INFINITY;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              float mb = -INFINITY;
              if (full_tile) {
#pragma unroll
                for (int k = 0; k < 16; k += 2) mb = fmax3(mb, sv[16 * h2 + k], sv[16 * h2 + k + 1]);
              } else {
                const int l = limb(2 * q + h2);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                  if (k < l) mb = fmaxf(mb, sv[16 * h2 + k]);
              }
              mx = fmaxf(mx, mb + (bias0(q, h2) + kmax));
            }
            return mx;
          } else {
            if (full_tile) {  // four independent chains
              float m4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
              for (int k = 4; k < 28; k += 8) {
                m4[0] = fmax3(m4[0], sv[k], sv[k + 1]);
                m4[1] = fmax3(m4[1], sv[k + 2], sv[k + 3]);
                m4[2] = fmax3(m4[2], sv[k + 4], sv[k + 5]);
                m4[3] = fmax3(m4[3], sv[k + 6], sv[k + 7]);
              }
              m4[0] = fmax3(m4[0], sv[28], sv[29]);
              m4[1] = fmax3(m4[1], sv[30], sv[31]);
              return fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
            }
            float mx = -INFINITY;
            const int l0 = limb(2 * q), l1 = limb(2 * q + 1);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if ((k & 15) < (k < 16 ? l0 : l1)) mx = fmaxf(mx, sv[k]);
            return mx;
          }
        };
        // Pass 1: row maximum, two chunks per TMEM wait (one where registers are short).
        float mx = -INFINITY;
        if constexpr (ALIBI || MIXED) {
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            float sv[32];
            tmem_ld32(tS + lane_base + 32 * q, sv);
            tmem_ld_wait(sv);
            mx = fmaxf(mx, chunk_max(sv, q));
          }
        } else {
#pragma unroll 1
          for (int q = 0; q < 4; q += 2) {
            float sv[32], sw[32];
            tmem_ld32(tS + lane_base + 32 * q, sv);
            tmem_ld32(tS + lane_base + 32 * (q + 1), sw);
            tmem_ld_wait(sv, sw);
            mx = fmax3(mx, chunk_max(sv, q), chunk_max(sw, q + 1));
          }
        }
        // Refresh the running maximum only when it grows by more than 2^8 (weights stay <= 256).
        float alpha = 1.f;
        if (mx > m_run + RESCALE_LOG2) {
          alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
          m_run = mx;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        // Rescale the running output when this row's maximum was refreshed (warp-uniform),
        // before any of this tile's P V; PV_t(g-1) has completed, since S_t(g) was issued
        // after it.
        if (j > j0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
        LAZY_PF_CLK(k2);
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
            const int l0 = limb(2 * q), l1 = limb(2 * q + 1);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if ((k & 15) >= (k < 16 ? l0 : l1)) sv[k] = -INFINITY;
          }
          // ALiBi: the bias moves into the subtrahend, m - b0 - slope (k & 15), stepped
          // by 2 slope from pair to pair of a block.
          uint64_t sub = mm, step2 = 0;
          if constexpr (ALIBI) step2 = f2(2.f * slope2, 2.f * slope2);
          uint32_t pw[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            if constexpr (ALIBI) {
              if ((k & 7) == 0) {
                const float b = m_use - bias0(q, k >> 3);
                sub = f2(b, b - slope2);
              } else {
                sub = f2_sub(sub, step2);
              }
            }
            const float2 dv = f2_split(f2_sub(f2(sv[2 * k], sv[2 * k + 1]), sub));
            const float e0 = ex2(dv.x), e1 = ex2(dv.y);
            pw[k] = pack_bf16x2(e0, e1);
            acc = f2_add(acc, f2(e0, e1));
          }
          tmem_st16(tS + lane_base + 16 * q, pw);
          if (q == 1) {  // the first 64 keys' P (and any rescaled O) are in TMEM
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_half[t]);
          }
        }
        const float2 sa = f2_split(acc);
        l_run = l_run * alpha + (sa.x + sa.y);
        LAZY_PF_CLK(k3);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        if (j + 1 < j1) {
          if (!warp_wait(&v_full[(g + 1) % NV], ((g + 1) / NV) & 1, a.status)) return ok = false;
          tm = read_mask((g + 1) % NV, iq, slope2, m_row);
        }
#ifdef LAZY_PREFILL_TRACE
        if (threadIdx.x == 0) {
          LAZY_PF_CLK(k4);
          LAZY_PF_COUNT(0, k1 - k0);
          LAZY_PF_COUNT(1, k2 - k1);
          LAZY_PF_COUNT(2, k3 - k2);
          LAZY_PF_COUNT(3, k4 - k3);
          LAZY_PF_COUNT(4, 1);
        }
#endif
      }
      pend = Pend{un, j0, j1, U0, gt - 1, sg, m_run, l_run, true};
      return true;
    });
    if (ok && pend.valid) ok = epilogue(pend);
    if (!ok) abort_flag = 1;
    LAZY_PF_TRACE(7, 7, global_timer_ns());
  }
  if constexpr (MIXED) mixed_combine(a, warp, THREADS / 32);
  tc_fence_before();
  __syncthreads();
  LAZY_PF_TRACE(7, 2, global_timer_ns());
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t launch_mixed(const MixedArgs& a, const CUtensorMap& qmap, const CUtensorMap& qmap_dec,
                         const CUtensorMap& kmap, const CUtensorMap& vmap, int grid, cudaStream_t st) {
  // a decode unit's 16-row groups each hold the query heads of one member: G % 16 == 0
  if (a.D != D || a.G % 16 != 0) return cudaErrorNotSupported;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.counters, 0, (size_t)(grid + 1) * 2 * BM * sizeof(int), st);
  if (e == cudaSuccess && a.B_dec > 0) e = cudaMemsetAsync(a.seq_done, 0, (size_t)a.B_dec * sizeof(int), st);
  if (e != cudaSuccess) return e;
  auto kern = prefill_stream_kernel<true, false, true>;
  e = set_smem_once<prefill_stream_kernel<true, false, true>>(SMEM);
  if (e != cudaSuccess) return e;
  // Cooperative: the decode merges wait for decode units of other CTAs, which must
  // therefore all be resident at once (one CTA per SM).
  MixedArgs ac = a;
  CUtensorMap mq = qmap, mk = kmap, mv = vmap, mqd = qmap_dec;
  void* args[] = {&ac, &mq, &mk, &mv, &mqd};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(THREADS), args, SMEM, st);
}

int prefill_stream_grid() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();
    return 152;
  }
  return sms;
}

size_t prefill_stream_counter_bytes(int grid) {
  return ((size_t)(grid + 1) * 2 * BM * sizeof(int) + 255) / 256 * 256;
}

size_t prefill_stream_workspace_bytes(int grid) {
  size_t bytes = prefill_stream_counter_bytes(grid) + (size_t)2 * grid * 2 * PARTIAL_TILE_FLOATS * sizeof(float);
#ifdef LAZY_PREFILL_TRACE
  bytes += (size_t)grid * 9 * 8 * 8;
#endif
  return bytes;
}

cudaError_t launch_prefill_stream(const PrefillArgs& a, bool lazy, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int grid, cudaStream_t st, const float* alibi) {
  if (a.D != D || a.G % 2 != 0) return cudaErrorNotSupported;
  if (a.B == 0 || a.max_q_len == 0 || grid <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.counters, 0, (size_t)(grid + 1) * 2 * BM * sizeof(int), st);
  if (e != cudaSuccess) return e;
  if (alibi) {
    e = set_smem_once<prefill_stream_kernel<false, true>>(SMEM);
    if (e != cudaSuccess) return e;
    PrefillAlibiArgs aa;
    static_cast<PrefillArgs&>(aa) = a;
    aa.alibi = alibi;
    prefill_stream_kernel<false, true><<<grid, THREADS, SMEM, st>>>(aa, qmap, kmap, vmap, qmap);
    return cudaGetLastError();
  }
  auto kern = lazy ? prefill_stream_kernel<true> : prefill_stream_kernel<false>;
  e = lazy ? set_smem_once<prefill_stream_kernel<true>>(SMEM) : set_smem_once<prefill_stream_kernel<false>>(SMEM);
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, SMEM, st>>>(a, qmap, kmap, vmap, qmap);  // (no decode units: qmap_dec unused)
  return cudaGetLastError();
}

}  // namespace lazy
