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
//   * a tile is 16 rows x 4 groups (1 KB of packed words).  Inside a CTA the
//     tiles of the current round are cut into 16 equal contiguous ranges, one
//     per warp; each warp streams its tiles through its own ring of shared
//     memory slots filled by TMA (64-byte swizzle: conflict-free reads), so
//     several kilobytes per warp are always in flight;
//   * partial sums go to shared memory, are combined over warps in warp
//     order, then over the cluster's CTAs in rank order through distributed
//     shared memory (deterministic: fixed summation order, no atomics).
// One pair of cluster barriers per round; most shapes need a single round.
// Every mbarrier wait is bounded: one that runs out sets a device error word.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace cg = cooperative_groups;

namespace q1 {

__device__ unsigned int g_narrow_err = 0;

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kQuad = 4;              // groups per tile
constexpr int kTileBytes = 16 * 64;   // 16 rows x 16 words
constexpr int kXsThreadStride = 80;   // bytes per (group, token, quad-thread) block of x'
constexpr int kSmemMax = 227 * 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// 1 / d_p and a_p of the bit-position encoding above.
__device__ __forceinline__ float inv_d(int p) {
  return p < 7 ? (float)(1 << (7 - p)) : (p == 7 ? 2.0f : (p < 15 ? (float)(1 << (15 - p)) : -0.5f));
}
__device__ __forceinline__ float a_of(int p) { return p == 7 ? 0.5f : 1.0f; }

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  // not volatile: no side effects, so the compiler may interleave the
  // independent MMA chains of a tile's four groups
  asm(
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

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false when it ran out (the device error word is set).
__device__ __noinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(addr, parity)) return true;
    if ((i & 15u) == 15u && globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(&g_narrow_err, 1u);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  if (mbar_try(addr, parity)) return true;
  return mbar_wait_bounded(addr, parity);
}

// Launch geometry, decided on the host.
struct Geo {
  int ks;     // CTAs per cluster (K slices)
  int nclus;  // clusters
  int tr;     // virtual row tiles per round
  int rpw;    // partial slots per warp (row tiles one warp can touch in a round)
  int ring;   // TMA slots per warp
};

struct SmemLayout {
  int ring, bars, xs, cs, part, red, meta, total;
};

// qmax: tiles (of 4 groups) per row tile in the widest K-slice; mst: tokens stored
__host__ __device__ inline SmemLayout smem_layout(int qmax, int mst, int tr, int rpw, int ring) {
  SmemLayout L;
  int off = 0;
  L.ring = off; off += kWarps * ring * kTileBytes;
  L.bars = off; off += align_up(kWarps * ring * 8, 128);
  // x' for qmax*4 groups x mst tokens, then one zero block (lanes with no token)
  L.xs = off; off += align_up((qmax * kQuad * mst + 1) * 4 * kXsThreadStride, 128);
  L.cs = off; off += align_up(qmax * kQuad * 8 * 8, 128);
  L.part = off; off += kWarps * rpw * 16 * 8 * 4;
  L.red = off; off += tr * 16 * 8 * 4;
  L.meta = off; off += align_up((kWarps + tr) * 4, 128);
  L.total = off + 1024;  // slack for aligning the dynamic shared memory base
  return L;
}

struct NarrowArgs {
  const uint16_t *s[2];
  const uint16_t *b[2];
  int64_t N;
  int K;
  int M;
  const __nv_bfloat16 *x;  // [M][K]
  __nv_bfloat16 *out;      // y [M][N] or h [M][N]
  Geo geo;
};

// Start of warp w's contiguous tile range when U tiles are cut into 16.
__host__ __device__ __forceinline__ int range_start(int U, int w) { return (U * w) / kWarps; }
// The warp whose range holds tile X (the last warp whose range starts at or before X).
__device__ __forceinline__ int warp_of_tile(int X, int U) {
  int w = (kWarps * (X + 1) + U - 1) / U - 1;
  return w < 0 ? 0 : (w > kWarps - 1 ? kWarps - 1 : w);
}

template <int NMAT, bool AFFINE>
__global__ void __launch_bounds__(kThreads, 1)
narrow_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
              NarrowArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA with the 64-byte swizzle wants 512-byte aligned slots: align the base
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  cg::cluster_group cluster = cg::this_cluster();

  const int M = a.M, K = a.K, G = K / 128;
  const Geo geo = a.geo;
  const int KS = geo.ks, RING = geo.ring;
  const int rank = (int)cluster.block_rank();
  const int clus = blockIdx.x / KS;
  const int g0 = (int)(((int64_t)rank * G) / KS), g1 = (int)(((int64_t)(rank + 1) * G) / KS);
  const int KSL = g1 - g0;
  const int Q = (KSL + kQuad - 1) / kQuad;  // tiles per row tile in this slice
  const int qmax = ((G + KS - 1) / KS + kQuad - 1) / kQuad;
  const SmemLayout L = smem_layout(qmax, M, geo.tr, geo.rpw, RING);
  unsigned char *ring = smem + L.ring;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
  unsigned char *xs = smem + L.xs;
  float2 *css = reinterpret_cast<float2 *>(smem + L.cs);  // [j][token]: (C or E, Sx)
  float *part = reinterpret_cast<float *>(smem + L.part);
  float *red = reinterpret_cast<float *>(smem + L.red);
  int *meta = reinterpret_cast<int *>(smem + L.meta);

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

  unsigned char *my_ring = ring + warp * RING * kTileBytes;
  uint64_t *my_bars = bars + warp * RING;
  if (lane < RING) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(my_bars + lane)) : "memory");
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();

  int round_v = v_lo;
  int T = min(geo.tr, v_hi - round_v);
  int U = T * Q;
  int ua = range_start(U, warp), ub = range_start(U, warp + 1);
  uint32_t issued = 0;  // tiles this warp consumed in earlier rounds (ring phase)

  // lane 0: TMA of the round's tile (row tile lv, quad q) into the slot of
  // sequence number `seq`
  auto issue = [&](int lv, int q, uint32_t seq) {
    const int vt = round_v + lv;
    const int mat = NMAT == 2 ? (vt & 1) : 0;
    const int rt = NMAT == 2 ? (vt >> 1) : vt;
    const int slot = (int)(seq % (uint32_t)RING);
    const uint32_t bar = smem_u32(my_bars + slot);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTileBytes)
                 : "memory");
    const CUtensorMap *tm = mat == 0 ? &tm0 : &tm1;
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(my_ring + slot * kTileBytes)), "l"(tm), "r"((g0 + q * kQuad) * 4), "r"(rt * 16),
        "r"(bar)
        : "memory");
  };
  auto prime = [&]() {  // first RING tiles of this warp's range
    if (lane == 0) {
      int lv = ua / Q, q = ua - (ua / Q) * Q;
      for (int i = 0; i < RING && ua + i < ub; ++i) {
        issue(lv, q, issued + (uint32_t)i);
        if (++q == Q) { q = 0; ++lv; }
      }
    }
  };
  prime();

  // the next kernel of a dependent chain may start streaming its weights now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // x may be the output of the preceding kernel: wait for it before reading
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- activation fragments of this CTA's K-slice -> shared memory, padded
  //      with zeros to whole tiles, plus the zero block for lanes gid >= M
  {
    const int jn = Q * kQuad;
    const int nitems = jn * M * 4;  // (j, m, t) blocks of 32 k
    for (int base = 0; base < nitems; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < nitems;
      const int tt = i & 3, jm = i >> 2;
      const int j = jm / M, m = jm - j * M;
      float c = 0.f, sx = 0.f;
      if (valid) {
        uint32_t pr[16];
        if (j < KSL) {
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
        css[j * 8 + m] = make_float2(AFFINE ? c : fmaf(0.5f, sx, c), sx);
      }
    }
    // zero block, and the (C, Sx) entries of tokens m >= M
    unsigned char *zb = xs + (size_t)jn * M * 4 * kXsThreadStride;
    for (int i = tid; i < 4 * kXsThreadStride / 16; i += kThreads)
      reinterpret_cast<uint4 *>(zb)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < jn * 8; i += kThreads)
      if ((i & 7) >= M) css[i] = make_float2(0.f, 0.f);
  }
  __syncthreads();

  // per-lane constants of the compute loop (32-bit shared-memory addresses)
  const uint32_t xlane = smem_u32(gid < M ? xs + ((size_t)gid * 4 + t) * kXsThreadStride
                                          : xs + ((size_t)Q * kQuad * M * 4 + t) * kXsThreadStride);
  const uint32_t xj_stride = gid < M ? (uint32_t)(M * 4 * kXsThreadStride) : 0u;  // per group
  const uint32_t clane = smem_u32(css + 2 * t);
  const uint32_t ring_lane = smem_u32(my_ring) + gid * 64 + 4 * t;
  const uint32_t part_lane = smem_u32(part) + (uint32_t)((gid * 8 + 2 * t) * 4);
  // word offsets of the four groups of a tile under the 64-byte swizzle (rows
  // gid and gid + 8 share it: ((r >> 1) & 3) is the same for both)
  const int swz = (gid >> 1) & 3;
  uint32_t woff[kQuad];
#pragma unroll
  for (int u = 0; u < kQuad; ++u) woff[u] = (uint32_t)((u ^ swz) << 4);

  while (true) {
    // ---- stream this warp's tiles [ua, ub) of the round
    const int vt_first = round_v + ua / Q;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    // scales (and biases) of one tile's 4 groups, rows gid and gid + 8; groups
    // past this K-slice (tile padding) read as scale 0
    auto load_meta = [&](int lv, int q, uint32_t (&sw)[kQuad], uint32_t (&bw)[kQuad]) {
      const int vt = round_v + lv;
      const int rt = NMAT == 2 ? (vt >> 1) : vt;
      const int mat = NMAT == 2 ? (vt & 1) : 0;
      const int rA = min(rt * 16 + gid, last_row), rB = min(rt * 16 + gid + 8, last_row);
      const int jb = q * kQuad;
      const size_t oA = (size_t)rA * G + g0 + jb, oB = (size_t)rB * G + g0 + jb;
      const uint16_t *pA = (mat == 0 ? a.s[0] : a.s[1]) + oA;
      const uint16_t *pB = (mat == 0 ? a.s[0] : a.s[1]) + oB;
      const uint16_t *Bp = mat == 0 ? a.b[0] : a.b[1];
      if (jb + kQuad <= KSL) {  // whole tile inside the K-slice (all but a slice's last tile)
#pragma unroll
        for (int u = 0; u < kQuad; ++u) {
          sw[u] = (uint32_t)__ldg(pA + u) | ((uint32_t)__ldg(pB + u) << 16);
          if (AFFINE) bw[u] = Bp ? ((uint32_t)__ldg(Bp + oA + u) | ((uint32_t)__ldg(Bp + oB + u) << 16))
                                 : 0xFFFFFFFFu;  // no stored bias: derive -s/2
        }
      } else {  // groups past the slice (tile padding) read as scale 0
#pragma unroll
        for (int u = 0; u < kQuad; ++u) {
          const bool in = jb + u < KSL;
          sw[u] = in ? ((uint32_t)__ldg(pA + u) | ((uint32_t)__ldg(pB + u) << 16)) : 0u;
          if (AFFINE)
            bw[u] = Bp ? (in ? ((uint32_t)__ldg(Bp + oA + u) | ((uint32_t)__ldg(Bp + oB + u) << 16)) : 0u)
                       : 0xFFFFFFFFu;
        }
      }
    };
    auto prefetch_meta_l2 = [&](int lv, int q) {
      const int vt = round_v + lv;
      const int rt = NMAT == 2 ? (vt >> 1) : vt;
      const uint16_t *Sp = (NMAT == 2 && (vt & 1)) ? a.s[1] : a.s[0];
      const int r = min(rt * 16 + (lane & 15), last_row);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(Sp + (size_t)r * G + g0 + q * kQuad));
    };
    uint32_t sw[kQuad], bw[kQuad], swn[kQuad], bwn[kQuad];
    // cursors (row tile, quad) of the current tile, the next one, and the one
    // RING ahead (the refill target), advanced without divisions
    int lv = ua / Q, q = ua - (ua / Q) * Q;
    int lv1 = lv, q1 = q;
    if (++q1 == Q) { q1 = 0; ++lv1; }
    int lvR = (ua + RING) / Q, qR = (ua + RING) - ((ua + RING) / Q) * Q;
    int slot = (int)(issued % (uint32_t)RING);
    uint32_t phase = (issued / (uint32_t)RING) & 1u;
    if (ua < ub) load_meta(lv, q, sw, bw);
    for (int tile = ua; tile < ub; ++tile) {
      const uint32_t seq = issued + (uint32_t)(tile - ua);
      const int vt = round_v + lv;
      const int jb = q * kQuad;
      if (tile + 1 < ub) load_meta(lv1, q1, swn, bwn);
      if (tile + RING < ub && lane < 16) prefetch_meta_l2(lvR, qR);
      const uint32_t tb = ring_lane + (uint32_t)(slot * kTileBytes);
      const uint32_t xb = xlane + (uint32_t)jb * xj_stride;
      // a wait that ran out has set the device error word; the results of this
      // call are then undefined, but the CTA still reaches its barriers
      mbar_wait(smem_u32(my_bars + slot), phase);
#pragma unroll
      for (int u = 0; u < kQuad; ++u) {
        const int j = jb + u;
        const uint32_t w0 = lds32(tb + woff[u]);
        const uint32_t w1 = lds32(tb + woff[u] + 8 * 64);
        uint32_t bfr[16];
        const uint32_t xu = xb + (uint32_t)u * xj_stride;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          uint4 v = lds128(xu + 16 * qq);
          bfr[4 * qq] = v.x; bfr[4 * qq + 1] = v.y; bfr[4 * qq + 2] = v.z; bfr[4 * qq + 3] = v.w;
        }
        const uint32_t w08 = w0 >> 8, w18 = w1 >> 8;
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
        const float4 cc = lds128f(clane + (uint32_t)j * 64);  // (C or E, Sx) of tokens 2t, 2t+1
        const float sa = __half2float(__ushort_as_half((uint16_t)(sw[u] & 0xFFFFu)));
        const float sb = __half2float(__ushort_as_half((uint16_t)(sw[u] >> 16)));
        if (AFFINE) {
          float ba, bb;
          if (bw[u] == 0xFFFFFFFFu) {  // matrix without stored biases: symmetric
            ba = __fmul_rn(-0.5f, sa);
            bb = __fmul_rn(-0.5f, sb);
          } else {
            ba = __half2float(__ushort_as_half((uint16_t)(bw[u] & 0xFFFFu)));
            bb = __half2float(__ushort_as_half((uint16_t)(bw[u] >> 16)));
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
#pragma unroll
      for (int u = 0; u < kQuad; ++u) {
        sw[u] = swn[u];
        if (AFFINE) bw[u] = bwn[u];
      }
      // the slot is free once every lane has read it: refill it RING tiles ahead
      __syncwarp();
      if (lane == 0 && tile + RING < ub) issue(lvR, qR, seq + (uint32_t)RING);
      // row tile finished (next tile belongs to another one, or range ends)
      if (tile + 1 == ub || lv1 != lv) {
        const uint32_t pp = part_lane + (uint32_t)((warp * geo.rpw + (vt - vt_first)) * 16 * 8 * 4);
        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(pp), "f"(acc[0]), "f"(acc[1]) : "memory");
        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(pp + 8 * 8 * 4), "f"(acc[2]), "f"(acc[3])
                     : "memory");
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
      }
      // advance the cursors and the ring position
      lv = lv1;
      q = q1;
      if (++q1 == Q) { q1 = 0; ++lv1; }
      if (++qR == Q) { qR = 0; ++lvR; }
      if (++slot == RING) { slot = 0; phase ^= 1u; }
    }
    issued += (uint32_t)(ub - ua);

    // ---- the next round's geometry
    const int next_v = round_v + T;
    int nT = 0, nU = 0, nua = 0, nub = 0;
    if (next_v < v_hi) {
      nT = min(geo.tr, v_hi - next_v);
      nU = nT * Q;
      nua = range_start(nU, warp);
      nub = range_start(nU, warp + 1);
    }
    __syncthreads();

    // ---- combine the warps' partials per row tile, in warp order.  The
    //      contributing warps of row tile lv and each warp's first row tile
    //      are computed once (meta[]), then every element sums its slots.
    if (tid < kWarps) {
      const int a0 = range_start(U, tid), a1 = range_start(U, tid + 1);
      meta[tid] = a0 < a1 ? a0 / Q : -1;
    }
    for (int lv = tid; lv < T; lv += kThreads)
      meta[kWarps + lv] = warp_of_tile(lv * Q, U) | (warp_of_tile(lv * Q + Q - 1, U) << 8);
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
    prime();
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
  cfg.dynamicSmemBytes = 96 * 1024;  // residency is bound by one CTA per SM anyway
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Packed words [N][K/32] as a 2-D uint32 tensor; boxes of 16 words x 16 rows
// with the 64-byte swizzle; rows >= N and words >= K/32 read as zero.
bool make_word_map(CUtensorMap *map, const uint32_t *w, int64_t N, int64_t K) {
  auto encode = encode_fn();
  if (!encode) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
  cuuint64_t gstride[1] = {(cuuint64_t)(K / 32) * 4};
  cuuint32_t box[2] = {16, 16};
  cuuint32_t estride[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(w), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NMAT, bool AFFINE>
cudaError_t launch_impl(NarrowArgs args, const uint32_t *w0, const uint32_t *w1, cudaStream_t st,
                        bool pdl) {
  auto kern = narrow_kernel<NMAT, AFFINE>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tm0, tm1;
  if (!make_word_map(&tm0, w0, args.N, args.K)) return cudaErrorInvalidValue;
  if (!make_word_map(&tm1, w1, args.N, args.K)) return cudaErrorInvalidValue;
  const int G = args.K / 128;
  const int M = args.M;
  const int NT = (int)((args.N + 15) / 16);
  // Pick the cluster size (K slices) that minimises the tiles of the busiest
  // CTA, ceil(row tiles per cluster) x ceil(tiles per slice), among those
  // whose shared memory fits; for it, the deepest TMA ring that fits.
  Geo best{};
  long best_cost = -1;
  for (int ks = 1; ks <= 8; ks *= 2) {
    if (ks > G) break;
    int nclus = max_clusters<NMAT, AFFINE>(ks);
    if (nclus > NT) nclus = NT;
    const int kslmax = (G + ks - 1) / ks, kslmin = G / ks;
    const int qmax = (kslmax + kQuad - 1) / kQuad, qmin = (kslmin + kQuad - 1) / kQuad;
    const int vmax = ((NT + nclus - 1) / nclus) * NMAT;
    for (int ring = 8; ring >= 3; --ring) {
      int tr = vmax, rpw = 0;
      bool ok = false;
      for (;;) {
        const int upw = (tr * qmax + kWarps - 1) / kWarps;  // tiles per warp, at most
        rpw = (upw + qmin - 1) / qmin + 1;
        if (smem_layout(qmax, M, tr, rpw, ring).total <= kSmemMax) { ok = true; break; }
        if (tr <= NMAT) break;
        tr = tr / 2;
        if (NMAT == 2) tr &= ~1;
        if (tr < NMAT) tr = NMAT;
      }
      if (!ok) continue;
      const int rounds = (vmax + tr - 1) / tr;
      // tiles of the busiest CTA, a round's two cluster barriers, and a shallow ring
      const long cost = (long)vmax * qmax * 4 + (long)rounds * 256 + (8 - ring) * 8;
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = Geo{ks, nclus, tr, rpw, ring};
      }
      break;  // deepest ring that fits for this ks
    }
  }
  if (best_cost < 0) return cudaErrorInvalidConfiguration;
  args.geo = best;
  const int qmax = ((G + best.ks - 1) / best.ks + kQuad - 1) / kQuad;
  const SmemLayout L = smem_layout(qmax, M, best.tr, best.rpw, best.ring);
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
  return cudaLaunchKernelEx(&cfg, kern, tm0, tm1, args);
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
  a.s[0] = a.s[1] = W.s;
  a.b[0] = a.b[1] = W.b;
  return W.b ? launch_impl<1, true>(a, W.w, W.w, st, pdl) : launch_impl<1, false>(a, W.w, W.w, st, pdl);
}

cudaError_t launch_narrow_gate_up(const WeightView &G, const WeightView &U, const void *x,
                                  int64_t M, void *h, cudaStream_t st, bool pdl) {
  NarrowArgs a = make_args(x, M, G.N, G.K, h);
  a.s[0] = G.s;
  a.s[1] = U.s;
  a.b[0] = G.b;
  a.b[1] = U.b;
  // With mixed metadata the affine variant runs for both matrices; it derives
  // -scale/2 for the one whose biases pointer is null.
  if (G.b || U.b) return launch_impl<2, true>(a, G.w, U.w, st, pdl);
  return launch_impl<2, false>(a, G.w, U.w, st, pdl);
}

unsigned int read_and_clear_narrow_errors(cudaStream_t st, cudaError_t *err) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_narrow_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_narrow_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (err) *err = e;
  return v;
}

}  // namespace q1
