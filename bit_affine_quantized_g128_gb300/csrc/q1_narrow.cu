// Narrow Q1 matmul: y[M][N] = x[M][K] . Wd^T for 1 <= M <= 8, with the
// weights kept packed (no dense temporary): the M = 1 decode product and the
// speculative-verifier windows of "Support Bonsai-27B affine Q1" (higgs PR
// #212), section "What" (narrow matrix multiplies of up to 8 flattened rows
// stay packed) and "Why" (point 3: a dense dequant per call allocated
// multi-GiB temporaries).  The fused FFN's gate/up half lives here too
// (section "What": fused dense-FFN operations).
//
// GB300 design.  The bound is the CUDA-core budget per weight, not only HBM:
// at ~6.7 TB/s and 1.125 bit/weight the GPU must retire ~4.7e13 weights/s,
// about one issue slot per weight.  So the MACs run on the tensor cores
// (mma.sync m16n8k16 bf16, 16 weight rows x 16 k x 8 tokens) and the unpack
// costs one LOP3 per two weights, whatever M is:
//
//   A register (two weights of one row) = (word & mask) | (1.0bf16x2 & ~mask)
//
// with the mask picking bits (p, p+16) of a word (or of word>>8).  The two
// bits land in the mantissa, the exponent lsb or the sign of two bf16 values
// whose base is 1.0, so each weight becomes a_p + d_p * q with constants
// (a_p, d_p) that depend only on the bit position p:
//   p = 0..6  : bits p, p+16 of word     -> 1 + 2^(p-7) q
//   p = 7     : bits 7, 23 (exponent lsb) -> 0.5 + 0.5 q
//   p = 8..14 : bits p-8, p+8 of word>>8  -> 1 + 2^(p-15) q
//   p = 15    : bits 15, 31 (sign)        -> 1 - 2 q
// The activations are pre-scaled by 1/d_p (a power of two, exact in bf16) and
// permuted into the same (p, p+16) pairs in shared memory by each CTA for its
// own K-slice, so one group of 128 k gives D = C_g + S1 with
// S1 = sum_{k in g} q_k x_k and C_g = sum a_p x'_k.  Per group and row:
//   symmetric: y += s * (D - C_g - Sx_g / 2)
//   affine   : y += s * (D - C_g) + b * Sx_g         (Sx_g = sum_{k in g} x_k)
// which is w = s*q + b summed over the group.
//
// Work decomposition (persistent: one 16-warp CTA per SM, all resident):
//   * a thread-block cluster of KS CTAs splits K into KS slices (CTA rank r
//     owns groups [G r / KS, G (r+1) / KS) and keeps their activation
//     fragments in shared memory for the whole kernel);
//   * the clusters split the 16-row tiles of W into contiguous ranges;
//   * inside a CTA, the (row tile, group) units of the current round are cut
//     into 16 equal contiguous ranges, one per warp, streamed through a
//     double-buffered register pipeline of up to 4 groups of one row tile;
//   * partial sums go to shared memory, are combined over warps in warp
//     order, then over the cluster's CTAs in rank order through distributed
//     shared memory (deterministic: fixed summation order, no atomics).
// One pair of cluster barriers per round; most shapes need a single round.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace cg = cooperative_groups;

namespace q1 {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 4;            // groups per register-pipeline stage
constexpr int kXsThreadStride = 80;  // bytes per (group, token, quad-thread) block of x'
constexpr int kSmemMax = 227 * 1024;

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// 1 / d_p and a_p of the bit-position encoding above.
__device__ __forceinline__ float inv_d(int p) {
  return p < 7 ? (float)(1 << (7 - p)) : (p == 7 ? 2.0f : (p < 15 ? (float)(1 << (15 - p)) : -0.5f));
}
__device__ __forceinline__ float a_of(int p) { return p == 7 ? 0.5f : 1.0f; }

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two weights (bits p and p+16 of `src`) -> bf16x2 with base 1.0: one LOP3
// selecting the masked bits of src and the other bits of `base` (the bf16x2
// pattern of (1.0, 1.0)), with the mask as the immediate.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t sel(uint32_t src, uint32_t base) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(r) : "r"(src), "n"(MASK), "r"(base));
  return r;
}
template <int P>
__device__ __forceinline__ uint32_t pair_reg(uint32_t w, uint32_t w8, uint32_t base) {
  if constexpr (P < 8) return sel<(0x00010001u << P)>(w, base);
  else if constexpr (P < 15) return sel<(0x00010001u << (P - 8))>(w8, base);
  else return sel<0x80008000u>(w, base);
}

// Launch geometry, decided on the host.
struct Geo {
  int ks;     // CTAs per cluster (K slices)
  int nclus;  // clusters
  int tr;     // virtual row tiles per round
  int rpw;    // partial slots per warp (row tiles one warp can touch in a round)
};

struct SmemLayout {
  int xs, cs, part, red, meta, total;
};

__host__ __device__ inline SmemLayout smem_layout(int kslmax, int tr, int rpw) {
  SmemLayout L;
  int off = 0;
  L.xs = off; off += align_up(kslmax * 8 * 4 * kXsThreadStride, 128);
  L.cs = off; off += align_up(kslmax * 8 * 8, 128);
  L.part = off; off += kWarps * rpw * 16 * 8 * 4;
  L.red = off; off += tr * 16 * 8 * 4;
  L.meta = off; off += align_up((kWarps + tr) * 4, 128);
  L.total = off;
  return L;
}

struct NarrowArgs {
  const uint32_t *w[2];
  const uint16_t *s[2];
  const uint16_t *b[2];
  int64_t N;
  int K;
  int M;
  const __nv_bfloat16 *x;  // [M][K]
  __nv_bfloat16 *out;      // y [M][N] or h [M][N]
  Geo geo;
};

// Start of warp w's contiguous unit range when U units are cut into 16.
__host__ __device__ __forceinline__ int range_start(int U, int w) { return (U * w) / kWarps; }
// The warp whose range holds unit X (the last warp whose range starts at or before X).
__device__ __forceinline__ int warp_of_unit(int X, int U) {
  int w = (kWarps * (X + 1) + U - 1) / U - 1;
  return w < 0 ? 0 : (w > kWarps - 1 ? kWarps - 1 : w);
}

// One register-pipeline stage: up to kChunk consecutive groups of one row tile.
struct Stage {
  uint32_t wa[kChunk], wb[kChunk];  // packed words, rows gid and gid+8
  uint32_t s[kChunk];               // fp16 scales: lo = row gid, hi = row gid+8
  uint32_t b[kChunk];               // fp16 biases (affine), same packing
  int vt, j0, n;                    // virtual row tile, first group (slice-local), units
};

template <int NMAT, bool AFFINE>
__global__ void __launch_bounds__(kThreads, 1) narrow_kernel(NarrowArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();

  const int M = a.M, K = a.K, G = K / 128, wpr = K / 32;
  const Geo geo = a.geo;
  const int KS = geo.ks;
  const int rank = (int)cluster.block_rank();
  const int clus = blockIdx.x / KS;
  const int g0 = (int)(((int64_t)rank * G) / KS), g1 = (int)(((int64_t)(rank + 1) * G) / KS);
  const int KSL = g1 - g0;
  const int kslmax = (G + KS - 1) / KS;
  const SmemLayout L = smem_layout(kslmax, geo.tr, geo.rpw);
  unsigned char *xs = smem + L.xs;
  float4 *css = reinterpret_cast<float4 *>(smem + L.cs);  // [j][token pair]: (C0, Sx0, C1, Sx1)
  float *part = reinterpret_cast<float *>(smem + L.part);
  float *red = reinterpret_cast<float *>(smem + L.red);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, t = lane & 3;
  const int NT = (int)((a.N + 15) / 16);
  const int last_row = (int)(a.N - 1);
  // this cluster's virtual row tiles (matrix = v % NMAT, row tile = v / NMAT)
  const int v_lo = (int)(((int64_t)NT * clus) / geo.nclus) * NMAT;
  const int v_hi = (int)(((int64_t)NT * (clus + 1)) / geo.nclus) * NMAT;

  // bf16x2 (1.0, 1.0), kept in one register for every unpack LOP3 (opaque to
  // the compiler, so that it is not re-materialised per instruction)
  uint32_t kbase;
  asm volatile("mov.b32 %0, 0x3F803F80;" : "=r"(kbase));

  int round_v = v_lo;
  int T = min(geo.tr, v_hi - round_v);
  int U = T * KSL;
  int ua = range_start(U, warp), ub = range_start(U, warp + 1);
  // loader cursor: next unit to load (as row tile + slice-local group) and units left
  int ld_vt = round_v + ua / KSL, ld_j = ua % KSL, ld_left = ub - ua;

  // Issue the loads of the next stage: consecutive groups of one row tile.
  // Rows beyond N read row N-1 (in bounds; their results are never stored).
  auto load_stage = [&](Stage &S) {
    const int n = min(kChunk, min(KSL - ld_j, ld_left));
    S.vt = ld_vt;
    S.j0 = ld_j;
    S.n = n;
    const int mat = NMAT == 2 ? (ld_vt & 1) : 0;
    const int rt = NMAT == 2 ? (ld_vt >> 1) : ld_vt;
    const int rA = min(rt * 16 + gid, last_row), rB = min(rt * 16 + gid + 8, last_row);
    const uint32_t *W = mat == 0 ? a.w[0] : a.w[1];
    const uint16_t *Sp = mat == 0 ? a.s[0] : a.s[1];
    const uint16_t *Bp = mat == 0 ? a.b[0] : a.b[1];
    const int g = g0 + ld_j;
    const uint32_t *pa = W + (size_t)rA * wpr + g * 4 + t;
    const uint32_t *pb = W + (size_t)rB * wpr + g * 4 + t;
    const uint16_t *sa = Sp + (size_t)rA * G + g;
    const uint16_t *sb = Sp + (size_t)rB * G + g;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (i < n) {
        S.wa[i] = __ldg(pa + 4 * i);
        S.wb[i] = __ldg(pb + 4 * i);
        S.s[i] = (uint32_t)__ldg(sa + i) | ((uint32_t)__ldg(sb + i) << 16);
        if (AFFINE) {
          if (Bp) {
            S.b[i] = (uint32_t)__ldg(Bp + (size_t)rA * G + g + i) |
                     ((uint32_t)__ldg(Bp + (size_t)rB * G + g + i) << 16);
          } else {
            S.b[i] = 0xFFFFFFFFu;  // no stored bias: derive -s/2
          }
        }
      }
    }
    ld_left -= n;
    ld_j += n;
    if (ld_j == KSL) {
      ld_j = 0;
      ++ld_vt;
    }
  };

  Stage SA, SB;
  // the first weights go out before anything else
  if (ld_left > 0) load_stage(SA);

  // the next kernel of a dependent chain may start streaming its weights now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // x may be the output of the preceding kernel: wait for it before reading
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- activation fragments of this CTA's K-slice -> shared memory, for 8
  //      tokens (rows m >= M are zero, so every lane loads unconditionally)
  {
    const int nitems = KSL * 8 * 4;  // (j, m, t) blocks of 32 k
    for (int base = 0; base < nitems; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < nitems;
      const int tt = i & 3, jm = i >> 2;
      const int j = jm >> 3, m = jm & 7;
      float c = 0.f, sx = 0.f;
      if (valid) {
        uint32_t pr[16];
        if (m < M) {
          const uint4 *src =
              reinterpret_cast<const uint4 *>(a.x + (size_t)m * K + (size_t)(g0 + j) * 128 + 32 * tt);
          uint32_t xv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = __ldg(src + q);
            xv[4 * q] = v.x; xv[4 * q + 1] = v.y; xv[4 * q + 2] = v.z; xv[4 * q + 3] = v.w;
          }
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            // x[p] is half (p & 1) of xv[p >> 1]; x[p+16] likewise in xv[8 + (p >> 1)]
            const uint32_t lo_bits = (p & 1) ? (xv[p >> 1] >> 16) : (xv[p >> 1] & 0xFFFFu);
            const uint32_t hi_bits = (p & 1) ? (xv[8 + (p >> 1)] >> 16) : (xv[8 + (p >> 1)] & 0xFFFFu);
            const float xl = __uint_as_float(lo_bits << 16), xh = __uint_as_float(hi_bits << 16);
            const float sc = inv_d(p);
            const float pl = xl * sc, ph = xh * sc;  // exact: power-of-two scaling
            const __nv_bfloat162 pb = __floats2bfloat162_rn(pl, ph);
            pr[p] = *reinterpret_cast<const uint32_t *>(&pb);
            c = fmaf(a_of(p), pl + ph, c);
            sx += xl + xh;
          }
        } else {
#pragma unroll
          for (int p = 0; p < 16; ++p) pr[p] = 0u;
        }
        uint4 *dst = reinterpret_cast<uint4 *>(xs + ((size_t)jm * 4 + tt) * kXsThreadStride);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pr[4 * q], pr[4 * q + 1], pr[4 * q + 2], pr[4 * q + 3]);
      }
      // the four quad blocks of one (j, m) sit in adjacent lanes
      c += __shfl_xor_sync(0xffffffffu, c, 1);
      sx += __shfl_xor_sync(0xffffffffu, sx, 1);
      c += __shfl_xor_sync(0xffffffffu, c, 2);
      sx += __shfl_xor_sync(0xffffffffu, sx, 2);
      if (valid && tt == 0) {
        // symmetric metadata folds the derived bias in: E = C + Sx / 2
        float *cf = reinterpret_cast<float *>(css) + (size_t)j * 16 + (m >> 1) * 4 + (m & 1) * 2;
        cf[0] = AFFINE ? c : fmaf(0.5f, sx, c);
        cf[1] = sx;
      }
    }
  }
  __syncthreads();

  while (true) {
    // ---- stream this warp's units [ua, ub) of the round, one stage at a time
    const int vt_first = round_v + ua / KSL;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto flush = [&](int vt) {
      float *pp = part + ((size_t)(warp * geo.rpw + (vt - vt_first)) * 16) * 8;
      pp[gid * 8 + 2 * t] = acc[0];
      pp[gid * 8 + 2 * t + 1] = acc[1];
      pp[(gid + 8) * 8 + 2 * t] = acc[2];
      pp[(gid + 8) * 8 + 2 * t + 1] = acc[3];
      acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    };
    auto compute_stage = [&](const Stage &S) {
      const unsigned char *xb = xs + ((size_t)(S.j0 * 8 + gid) * 4 + t) * kXsThreadStride;
      const float4 *cb = css + (size_t)S.j0 * 4 + t;
#pragma unroll
      for (int i = 0; i < kChunk; ++i) {
        if (i < S.n) {
          uint32_t bfr[16];
          const uint4 *src = reinterpret_cast<const uint4 *>(xb + (size_t)i * 8 * 4 * kXsThreadStride);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v = src[q];
            bfr[4 * q] = v.x; bfr[4 * q + 1] = v.y; bfr[4 * q + 2] = v.z; bfr[4 * q + 3] = v.w;
          }
          const uint32_t w0 = S.wa[i], w1 = S.wb[i], w08 = w0 >> 8, w18 = w1 >> 8;
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t af[4];
#define Q1_MMA_STEP(JJ)                              \
  af[0] = pair_reg<2 * (JJ)>(w0, w08, kbase);        \
  af[1] = pair_reg<2 * (JJ)>(w1, w18, kbase);        \
  af[2] = pair_reg<2 * (JJ) + 1>(w0, w08, kbase);    \
  af[3] = pair_reg<2 * (JJ) + 1>(w1, w18, kbase);    \
  mma_bf16_16816(d, af, bfr[2 * (JJ)], bfr[2 * (JJ) + 1]);
          Q1_MMA_STEP(0) Q1_MMA_STEP(1) Q1_MMA_STEP(2) Q1_MMA_STEP(3)
          Q1_MMA_STEP(4) Q1_MMA_STEP(5) Q1_MMA_STEP(6) Q1_MMA_STEP(7)
#undef Q1_MMA_STEP
          const float4 cc = cb[(size_t)i * 4];  // (C or E, Sx) of tokens 2t, 2t+1
          const float sa = __half2float(__ushort_as_half((uint16_t)(S.s[i] & 0xFFFFu)));
          const float sb = __half2float(__ushort_as_half((uint16_t)(S.s[i] >> 16)));
          if (AFFINE) {
            float ba, bb;
            if (S.b[i] == 0xFFFFFFFFu) {  // matrix without stored biases: symmetric
              ba = __fmul_rn(-0.5f, sa);
              bb = __fmul_rn(-0.5f, sb);
            } else {
              ba = __half2float(__ushort_as_half((uint16_t)(S.b[i] & 0xFFFFu)));
              bb = __half2float(__ushort_as_half((uint16_t)(S.b[i] >> 16)));
            }
            acc[0] = fmaf(sa, d[0] - cc.x, fmaf(ba, cc.y, acc[0]));
            acc[1] = fmaf(sa, d[1] - cc.z, fmaf(ba, cc.w, acc[1]));
            acc[2] = fmaf(sb, d[2] - cc.x, fmaf(bb, cc.y, acc[2]));
            acc[3] = fmaf(sb, d[3] - cc.z, fmaf(bb, cc.w, acc[3]));
          } else {
            acc[0] = fmaf(sa, d[0] - cc.x, acc[0]);
            acc[1] = fmaf(sa, d[1] - cc.z, acc[1]);
            acc[2] = fmaf(sb, d[2] - cc.x, acc[2]);
            acc[3] = fmaf(sb, d[3] - cc.z, acc[3]);
          }
        }
      }
    };
    // two stages in flight: load the next while computing the current
    bool have_a = ua < ub, have_b = false;
    while (have_a || have_b) {
      if (have_a) {
        have_b = ld_left > 0;
        if (have_b) load_stage(SB);
        compute_stage(SA);
        if (!have_b || SB.vt != SA.vt) flush(SA.vt);
        have_a = false;
      }
      if (have_b) {
        have_a = ld_left > 0;
        if (have_a) load_stage(SA);
        compute_stage(SB);
        if (!have_a || SA.vt != SB.vt) flush(SB.vt);
        have_b = false;
      }
    }

    // ---- the next round's geometry, and its first stage of weights in flight
    const int next_v = round_v + T;
    int nT = 0, nU = 0, nua = 0, nub = 0;
    if (next_v < v_hi) {
      nT = min(geo.tr, v_hi - next_v);
      nU = nT * KSL;
      nua = range_start(nU, warp);
      nub = range_start(nU, warp + 1);
      ld_vt = next_v + nua / KSL;
      ld_j = nua % KSL;
      ld_left = nub - nua;
      if (ld_left > 0) load_stage(SA);
    }
    __syncthreads();

    // ---- combine the warps' partials per row tile, in warp order.  The
    //      contributing warps of row tile lv and each warp's first row tile
    //      are computed once (meta[]), then every element sums its slots.
    int *meta = reinterpret_cast<int *>(smem + L.meta);  // [0,16): first lv per warp (-1 empty); [16..): wf | wl << 8
    if (tid < kWarps) {
      const int a0 = range_start(U, tid), a1 = range_start(U, tid + 1);
      meta[tid] = a0 < a1 ? a0 / KSL : -1;
    }
    for (int lv = tid; lv < T; lv += kThreads)
      meta[kWarps + lv] = warp_of_unit(lv * KSL, U) | (warp_of_unit(lv * KSL + KSL - 1, U) << 8);
    __syncthreads();
    for (int i = tid; i < T * 128; i += kThreads) {
      const int lv = i >> 7, e = i & 127;
      const int fl = meta[kWarps + lv];
      float sum = 0.f;
      for (int w = fl & 0xFF; w <= (fl >> 8); ++w) {
        const int f = meta[w];
        if (f < 0) continue;  // empty range: this warp wrote nothing
        sum += part[((size_t)(w * geo.rpw + (lv - f)) * 16) * 8 + e];
      }
      red[(size_t)lv * 128 + e] = sum;
    }
    cluster.sync();

    // ---- cluster reduction in rank order; rank r finishes 1/KS of the row tiles
    {
      int lo, hi;
      if (NMAT == 2) {  // (gate, up) pairs of one row tile are adjacent: whole pairs per rank
        const int pp = (T / 2 + KS - 1) / KS;
        lo = min(T, rank * pp * 2);
        hi = min(T, lo + pp * 2);
      } else {
        const int per = (T + KS - 1) / KS;
        lo = min(T, rank * per);
        hi = min(T, lo + per);
      }
      const int cnt = ((hi - lo) / NMAT) * 16 * M;
      for (int i = tid; i < cnt; i += kThreads) {
        const int lv = lo + (i / (16 * M)) * NMAT, r = (i / M) % 16, m = i % M;
        const int64_t rt = (round_v + lv) / NMAT;
        const int64_t n = rt * 16 + r;
        if (n >= a.N) continue;
        float v0 = 0.f, v1 = 0.f;
        for (int q = 0; q < KS; ++q) {
          const float *rq = cluster.map_shared_rank(red, q);
          v0 += rq[(size_t)lv * 128 + r * 8 + m];
          if (NMAT == 2) v1 += rq[(size_t)(lv + 1) * 128 + r * 8 + m];
        }
        float o = v0;
        if (NMAT == 2) o = v0 / (1.0f + expf(-v0)) * v1;  // SiLU(gate) * up
        a.out[(size_t)m * a.N + n] = __float2bfloat16_rn(o);
      }
    }
    cluster.sync();  // every rank is done reading this round's partials

    if (next_v >= v_hi) break;
    round_v = next_v;
    T = nT;
    U = nU;
    ua = nua;
    ub = nub;
  }
}

// ---------------------------------------------------------------------------
// host: geometry
// ---------------------------------------------------------------------------
int sm_count_cached() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int NMAT, bool AFFINE>
int max_clusters(int ks) {
  static int cache[9] = {0};
  if (cache[ks]) return cache[ks];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ks * 64), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 96 * 1024;  // a typical footprint; residency is bound by 1 CTA/SM anyway
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)ks;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, narrow_kernel<NMAT, AFFINE>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count_cached() / ks;
  }
  if (n < 1) n = 1;
  cache[ks] = n;
  return n;
}

template <int NMAT, bool AFFINE>
cudaError_t launch_impl(NarrowArgs args, cudaStream_t st, bool pdl) {
  auto kern = narrow_kernel<NMAT, AFFINE>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int G = args.K / 128;
  const int NT = (int)((args.N + 15) / 16);
  // Pick the cluster size (K slices) that minimises the units of the busiest
  // CTA: ceil(row tiles per cluster) x ceil(groups per slice), among those
  // whose shared memory fits.
  Geo best{};
  long best_cost = -1;
  for (int ks = 1; ks <= 8; ks *= 2) {
    if (ks > G) break;
    int nclus = max_clusters<NMAT, AFFINE>(ks);
    if (nclus > NT) nclus = NT;
    const int kslmax = (G + ks - 1) / ks, kslmin = G / ks;
    const int vmax = ((NT + nclus - 1) / nclus) * NMAT;
    const int xs_bytes = align_up(kslmax * 8 * 4 * kXsThreadStride, 128) + align_up(kslmax * 8 * 8, 128);
    int tr = vmax, rpw = 0;
    bool ok = false;
    for (;;) {
      const int upw = (tr * kslmax + kWarps - 1) / kWarps;  // units per warp, at most
      rpw = (upw + kslmin - 1) / kslmin + 1;
      const int total = xs_bytes + kWarps * rpw * 512 + tr * 512 + align_up((kWarps + tr) * 4, 128);
      if (total <= kSmemMax) { ok = true; break; }
      if (tr <= NMAT) break;
      tr = tr / 2;
      if (NMAT == 2) tr &= ~1;
      if (tr < NMAT) tr = NMAT;
    }
    if (!ok) continue;
    const int rounds = (vmax + tr - 1) / tr;
    const long cost = (long)vmax * kslmax + (long)rounds * 64;  // a round costs ~2 cluster barriers
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = Geo{ks, nclus, tr, rpw};
    }
  }
  if (best_cost < 0) return cudaErrorInvalidConfiguration;
  args.geo = best;
  const SmemLayout L = smem_layout((G + best.ks - 1) / best.ks, best.tr, best.rpw);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(best.nclus * best.ks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = (unsigned)best.ks;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

NarrowArgs make_args(const void *x, int64_t M, int64_t N, int64_t K, void *out) {
  NarrowArgs a = {};
  a.x = static_cast<const __nv_bfloat16 *>(x);
  a.N = N;
  a.K = (int)K;
  a.M = (int)M;
  a.out = static_cast<__nv_bfloat16 *>(out);
  return a;
}

}  // namespace

cudaError_t launch_narrow(const WeightView &W, const void *x, int64_t M, void *y,
                          cudaStream_t st, bool pdl) {
  NarrowArgs a = make_args(x, M, W.N, W.K, y);
  a.w[0] = a.w[1] = W.w;
  a.s[0] = a.s[1] = W.s;
  a.b[0] = a.b[1] = W.b;
  return W.b ? launch_impl<1, true>(a, st, pdl) : launch_impl<1, false>(a, st, pdl);
}

cudaError_t launch_narrow_gate_up(const WeightView &G, const WeightView &U, const void *x,
                                  int64_t M, void *h, cudaStream_t st, bool pdl) {
  NarrowArgs a = make_args(x, M, G.N, G.K, h);
  a.w[0] = G.w;
  a.w[1] = U.w;
  a.s[0] = G.s;
  a.s[1] = U.s;
  a.b[0] = G.b;
  a.b[1] = U.b;
  // With mixed metadata the affine variant runs for both matrices; it derives
  // -scale/2 for the one whose biases pointer is null.
  if (G.b || U.b) return launch_impl<2, true>(a, st, pdl);
  return launch_impl<2, false>(a, st, pdl);
}

}  // namespace q1
