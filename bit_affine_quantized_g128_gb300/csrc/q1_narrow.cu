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
// The activations are scaled by 1/d_p (a power of two: exact) and paired as
// (x_p, x_{p+16}), so one group of 128 k gives D = C_g + S1 with
// S1 = sum_{k in g} q_k x_k and C_g = sum a_p x'_k.  Per group and row:
//   symmetric: y += s * (D - E_g),  E_g = C_g + Sx_g / 2
//   affine   : y += s * (D - C_g) + b * Sx_g         (Sx_g = sum_{k in g} x_k)
// which is w = s*q + b summed over the group.  C_g and Sx_g / 2 come from the
// tensor cores too: one MMA chain per group whose A rows 0..7 hold the a_p
// pattern and rows 8..15 hold d_p / 2 (all exact in bf16); -E_g (or -C_g) is
// then the accumulator that the group's MMA chain starts from.
//
// Work decomposition (one CTA per SM: up to 8 consumer warps and one
// producer warp):
//   * K is cut into spans of 4 groups (512 k).  A thread-block cluster of KS
//     CTAs splits the spans into KS contiguous slices; inside a CTA every
//     consumer warp owns one span for the whole launch, and with 9 or 10
//     spans on 8 warps (5 on 4) also one group of the remaining spans, so
//     that the SM's four sub-partitions get equal work; a warp keeps the
//     activation fragments of its 4 or 5 groups (16 registers each) and their
//     C/E terms in registers;
//   * the clusters split the 16-row tiles of W into contiguous ranges; the
//     R warps that own the same span take every R-th row tile of the range;
//   * the producer warp streams the CTA's row tiles, in order, through a
//     ring of row-tile slots: per slot the words as 1 KB per span (16 rows x
//     16 words, 64-byte swizzle: conflict-free reads), one 3-D TMA box for
//     all the CTA's spans when K % 512 == 0 (else one 2-D box per span), and
//     one box with the 16 rows' scales (and biases) of the whole K-slice, all
//     completing on the slot's mbarrier; the consumers hand the slot back
//     through a second mbarrier;
//   * the groups' MMA chains of a tile are interleaved, so that a warp
//     always has four or five independent MMAs in flight;
//   * per-tile partial sums go to shared memory and are combined over the
//     spans in a fixed order, then over the cluster's CTAs in rank order
//     through distributed shared memory (deterministic, no atomics).
// Every mbarrier wait is bounded: one that runs out sets a device error word.
#include <cooperative_groups.h>
#include <type_traits>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace cg = cooperative_groups;

namespace q1 {

__device__ unsigned int g_narrow_err = 0;
// Diagnostics (set from the host between launches): the limit of every
// bounded wait, and a switch that makes the producers issue nothing, so that
// every wait for their data runs out (no copy is then in flight).
__constant__ unsigned long long c_narrow_wait_ns = 2000000000ull;
__constant__ int c_narrow_stall = 0;

namespace {

constexpr int kMaxSpans = 10;                     // spans per CTA
constexpr int kMaxWarps = 8;                      // consumer warps
constexpr int kMaxThreads = (kMaxWarps + 1) * 32;  // + the producer warp
constexpr int kQuad = 4;                          // groups per span
constexpr int kMaxKS = 8;                         // CTAs per cluster (K slices)
constexpr int kTileBytes = 16 * 64;               // 16 rows x 16 words
constexpr int kSmemMax = 227 * 1024;
constexpr int kRingBytes = 24 * 1024;             // ring slots per SM, in bytes (about)

// Consumer warps along K for a CTA of qs spans.  Each warp owns one span,
// except that 9 or 10 spans go to 8 warps and 5 spans to 4 warps; the spans
// past the warps are then dealt out one group per warp (warp w also takes
// group w % 4 of span nw + w / 4).  The warps are spread round-robin over the
// SM's four sub-partitions, whose tensor and integer pipes bound the tile
// loop: 10 one-span warps would load two sub-partitions with three warps
// (12 groups) while the other two carry 8; 8 warps of 5 groups load each
// with 10.
__host__ __device__ inline int kwarps(int qs) { return qs > 8 ? 8 : (qs == 5 ? 4 : qs); }

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// bf16 bit patterns (both halves) of the encoding constants
constexpr uint32_t bf16_pow2(int e) { return (uint32_t)(e + 127) << 7; }
constexpr uint32_t dup2(uint32_t h) { return h | (h << 16); }
constexpr uint32_t inv_d_bits(int p) {  // 1 / d_p
  return dup2(p < 7 ? bf16_pow2(7 - p)
                    : p == 7 ? bf16_pow2(1) : p < 15 ? bf16_pow2(15 - p) : (0x8000u | bf16_pow2(-1)));
}
constexpr uint32_t a_bits(int p) { return dup2(p == 7 ? bf16_pow2(-1) : bf16_pow2(0)); }  // a_p
constexpr uint32_t halfd_bits(int p) {                                                   // d_p / 2
  return dup2(p < 7 ? bf16_pow2(p - 8)
                    : p == 7 ? bf16_pow2(-2) : p < 15 ? bf16_pow2(p - 16) : (0x8000u | bf16_pow2(0)));
}

__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  // not volatile: no side effects, so the compiler may interleave the
  // independent MMA chains of a tile's four groups
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// first MMA of a chain: accumulator input c, output d
__device__ __forceinline__ void mma_from(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
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

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}
// bf16x2 a * b, exact for a power-of-two b (the -0 addend keeps signs of zeros)
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

// (lo, hi) -> bf16x2, each rounded to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// Two weights (bits q and q+16 of `src`) -> bf16x2 with base 1.0, the mask in
// a register (the small-group mapping's masks depend on the lane).
__device__ __forceinline__ uint32_t selr(uint32_t src, uint32_t mask, uint32_t base) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(r) : "r"(src), "r"(mask), "r"(base));
  return r;
}
// activations i, i+1 of x (dtype xdt) as bf16x2, rounded once for fp16/fp32
__device__ __forceinline__ uint32_t x_pair(const void *x, int xdt, size_t i) {
  if (xdt == Q1_F32) {
    const float2 v = __ldg(reinterpret_cast<const float2 *>(static_cast<const float *>(x) + i));
    return pack_bf16x2(v.x, v.y);
  }
  const uint32_t v = __ldg(reinterpret_cast<const unsigned int *>(static_cast<const uint16_t *>(x) + i));
  if (xdt == Q1_F16) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&v));
    return pack_bf16x2(f.x, f.y);
  }
  return v;
}

// One of the two fp16 or bf16 metadata values packed in `pair` (hi: the upper
// one) widened to fp32, exactly.  For fp16 this is the FMA pipe's half-to-float
// conversion reading the chosen half in place (no shift on the integer pipe,
// which the unpack keeps busy).
__device__ __forceinline__ float meta_half_f32(uint32_t pair, int hi, bool bf16) {
  if (bf16) return __uint_as_float(hi ? (pair & 0xFFFF0000u) : (pair << 16));
  const __half2 h2 = *reinterpret_cast<const __half2 *>(&pair);
  return hi ? __high2float(h2) : __low2float(h2);
}

// one output value in the activation dtype (one rounding for 16-bit types)
__device__ __forceinline__ void store_act(void *out, size_t i, float v, int dt) {
  if (dt == Q1_F32) static_cast<float *>(out)[i] = v;
  else if (dt == Q1_F16) static_cast<__half *>(out)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
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
// Bounded wait, all inline (no call in the tile loop): false when it ran out
// (the device error word is set).  Each wait runs out on its own limit: a
// check of the error word in the polling loop cost 1.3 % on the decode step.
__device__ __forceinline__ bool mbar_wait(uint32_t addr, uint32_t parity) {
  if (mbar_try(addr, parity)) return true;
  const unsigned long long t0 = globaltimer();
#pragma unroll 1
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(addr, parity)) return true;
    if ((i & 15u) == 0u && globaltimer() - t0 > c_narrow_wait_ns) {
      atomicOr(&g_narrow_err, 1u);
      return false;
    }
  }
}

// Launch geometry, decided on the host.
struct Geo {
  int ks;     // CTAs per cluster (K slices)
  int nclus;  // clusters
  int qm;     // span slots per CTA (spans of the widest slice)
  int R;      // consumer warps per span (row-tile interleave)
  int tr;     // virtual row tiles per round
  int ring;   // ring slots (row tiles in flight) per CTA
  int mst;    // tokens stored per partial row (1, 2, 4 or 8)
};

// metadata row of a slot: the groups of spans (q_lo & ~1) .. q_lo + qm, in
// whole boxes of 8 groups; gps = groups per span of 512 k (4 for groups of
// 128 weights, 8 for 64, 16 for 32)
__host__ __device__ inline int meta_groups(int qm, int gps = 4) { return (gps * (qm + 1) + 7) / 8 * 8; }

// Warps that hold 5 groups of 128 k, the most any warp holds (kwarps).
constexpr int kMaxUnits = 5;

struct SmemLayout {
  int ring, meta, bars, part, red, seeds, total;
  int slot_words, slot_meta;  // bytes per ring slot
};

// gw: words of 32 weights per metadata group (4, 2 or 1).  Groups of 64 or 32
// weights keep their accumulator seeds in shared memory: per consumer warp,
// unit of 128 k and group, a float4 for each of the quad's four lanes.
__host__ __device__ inline SmemLayout smem_layout(const Geo &g, bool affine, int gw = 4) {
  SmemLayout L;
  L.slot_words = g.qm * kTileBytes;
  L.slot_meta = align_up(16 * meta_groups(g.qm, 16 / gw) * 2 * (affine ? 2 : 1), 128);
  int off = 0;
  L.ring = off; off += g.ring * L.slot_words;
  L.meta = off; off += g.ring * L.slot_meta;
  L.bars = off; off += align_up(2 * g.ring * 8, 128);
  L.part = off; off += g.tr * kwarps(g.qm) * 16 * (g.mst < 2 ? 2 : g.mst) * 4;
  L.red = off; off += g.ks > 1 ? g.tr * 16 * (g.mst < 2 ? 2 : g.mst) * 4 : 0;
  L.seeds = off; off += gw < 4 ? kwarps(g.qm) * g.R * kMaxUnits * (4 / gw) * 64 : 0;
  L.total = off + 1024;  // slack for aligning the dynamic shared memory base
  return L;
}

struct NarrowArgs {
  const uint16_t *s[2];
  const uint16_t *b[2];
  int64_t N;
  int K;
  int M;
  const void *x;  // [M][K], xdt
  void *out;      // y [M][N] or h [M][N], ydt
  int xdt, ydt;   // q1_dtype of x and of the output
  Geo geo;
  // strides of the shared-memory layout, computed on the host so that the
  // tile loop reads them as constants
  int slot_words, slot_meta, part_tile;
  int meta_bf16;  // bit m: matrix m's scales/biases are bf16 (else fp16)
  int w3;         // the w3 maps are set: one TMA per slot for the words
};

// Tensor maps of the (up to two) matrices: packed words, scales, biases.
// w3[m][v]: the same words as a 3-D tensor (16 words of a span, rows, spans),
// so that one box of 16 rows x (qm - v) spans fills a whole ring slot.
struct Maps {
  CUtensorMap w[2], s[2], b[2];
  CUtensorMap w3[2][2];
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Cluster barrier without release semantics.  It closes a round of remote
// reads: those values are already in registers (every one has been summed
// and stored), so nothing needs to become visible, and the arrival does not
// wait for this thread's outstanding global stores as a releasing one would.
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// One CTA: NC = kwarps(qm) * R consumer warps and one producer warp (the
// last).  The producer streams the CTA's row tiles in order through a ring
// of row-tile slots: per slot 1 KB of words per span of the CTA (16 rows x
// 16 words, 64-byte swizzle) and the rows' metadata.  Consumer warp
// (qi, ri) owns span q_lo + qi, plus one group of a span past the K-warps
// when the CTA has more spans than K-warps, and takes the row tiles ri,
// ri + R, ... of each round.
// FASTMETA: G % 8 == 0 and 16-byte aligned metadata, so the scales (and
// biases) come as one TMA box of meta_groups(qm) groups x 16 rows; otherwise
// the producer's lanes load them (zero past K) and store them before their
// arrivals.  Either way a slot's metadata is [16 rows][meta_groups] fp16
// starting at group 4 (q_lo & ~1).
// GW: words of 32 weights per metadata group, 4 (groups of 128), 2 (64) or 1
// (32).  With 4 every m16n8k16 step of a lane pairs word t of its group with
// the other lanes' words, so one step spans a whole group.  With 2 or 1 a step
// must stay within one group: the quad's four lanes then take different bit
// pairs of one word (lane t the pairs 2t and 2t + 1 of each half), which
// closes a chain of MMAs on every group; the group's accumulator seeds (C_g
// or E_g, and Sx_g) go to a shared-memory table, since a warp holds up to 20
// groups.
template <int NMAT, bool AFFINE, bool FASTMETA, int VAR, int GW>
__global__ void __launch_bounds__(kMaxThreads, 1)
narrow_kernel(const __grid_constant__ Maps maps, NarrowArgs a) {
  static_assert(GW == 4 || GW == 2 || GW == 1, "words per metadata group");
  constexpr int GPS = 16 / GW;  // metadata groups per span of 512 k
  constexpr int GPU = 4 / GW;   // metadata groups per unit of 128 k
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA with the 64-byte swizzle wants 512-byte aligned boxes: align the base
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  cg::cluster_group cluster = cg::this_cluster();

  const int M = a.M, K = a.K, G = K / 128;  // G: units of 128 k
  const int GM = K / (32 * GW);               // metadata groups per row
  const int64_t N = a.N;
  const Geo geo = a.geo;
  const int KS = geo.ks, RING = geo.ring, QM = geo.qm, R = geo.R, TR = geo.tr;
  const int MST = geo.mst < 2 ? 2 : geo.mst;  // tokens stored per partial row (a lane stores a pair)
  const SmemLayout L = smem_layout(geo, AFFINE, GW);
  const int NWM = kwarps(QM);               // K-warps of the widest slice
  const int NC = NWM * R;                   // consumer warps
  const int MROW = meta_groups(QM, GPS) * 2;  // bytes per metadata row

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, t = lane & 3;
  const int rank = (int)cluster.block_rank();
  const int clus = blockIdx.x / KS;
  const int QK = (G + kQuad - 1) / kQuad;  // spans in K
  const int q_lo = (int)(((int64_t)QK * rank) / KS), q_hi = (int)(((int64_t)QK * (rank + 1)) / KS);
  const int QS = q_hi - q_lo;               // spans of this CTA
  const int NW = kwarps(QS);                // K-warps of this CTA
  const int q_base = q_lo & ~1;             // first span of the metadata rows
  const int NT = (int)((N + 15) / 16);
  const int v_lo = (int)(((int64_t)NT * clus) / geo.nclus) * NMAT;
  const int v_hi = (int)(((int64_t)NT * (clus + 1)) / geo.nclus) * NMAT;

  const uint32_t ring_s = smem_u32(smem + L.ring);
  const uint32_t meta_s = smem_u32(smem + L.meta);
  const uint32_t full_s = smem_u32(smem + L.bars);  // full[RING], then empty[RING]
  const uint32_t empty_s = full_s + 8 * RING;
  float *part = reinterpret_cast<float *>(smem + L.part);
  float *red = reinterpret_cast<float *>(smem + L.red);

  if (warp == NC && lane < RING) {
    // full: the producer's expect_tx (plus, without metadata TMA, the 32
    // producer lanes' arrivals); empty: one arrival per K-warp
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full_s + 8 * lane), "r"(FASTMETA ? 1 : 33)
                 : "memory");
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty_s + 8 * lane), "r"(NW) : "memory");
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  // the next kernel of a dependent chain may start streaming its weights now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == NC) {
    // ================= producer =================
    const int nv = v_hi - v_lo;
    int j = 0;
    uint32_t slot = 0, ph = 0;
    auto issue_next = [&]() {
      const int v = v_lo + j;
      const int mat = NMAT == 2 ? (v & 1) : 0;
      const int rt = NMAT == 2 ? (v >> 1) : v;
      const bool has_b = AFFINE && (mat ? a.b[1] : a.b[0]) != nullptr;
      const uint32_t fb = full_s + 8 * slot;
      // the slot's previous tile has been read by its consumer warps
      mbar_wait(empty_s + 8 * slot, ph ^ 1u);
      // (diagnostics) a stalled producer issues nothing: the slot's full
      // barrier never completes and the consumers' waits run out
      if (!c_narrow_stall) {
        const uint32_t mdst = meta_s + slot * L.slot_meta;
        if (lane == 0) {
          const uint32_t bytes =
              QS * kTileBytes + (FASTMETA ? (uint32_t)(16 * MROW) * (has_b ? 2u : 1u) : 0u);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
          const CUtensorMap *wm = mat ? &maps.w[1] : &maps.w[0];
          const uint32_t wdst = ring_s + slot * L.slot_words;
          if (a.w3) {
            // one box: 16 words x 16 rows x QS spans, laid out span by span as
            // the per-span boxes would be
            const CUtensorMap *wm3 = &maps.w3[mat][QS == QM ? 0 : 1];
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
                "[%5];" ::"r"(wdst),
                "l"(wm3), "r"(0), "r"(rt * 16), "r"(q_lo), "r"(fb)
                : "memory");
          } else {
            for (int qs = 0; qs < QS; ++qs) tma_2d(wdst + qs * kTileBytes, wm, (q_lo + qs) * 16, rt * 16, fb);
          }
          if (FASTMETA) {
            tma_2d(mdst, mat ? &maps.s[1] : &maps.s[0], q_base * GPS, rt * 16, fb);
            if (has_b) tma_2d(mdst + 16 * MROW, mat ? &maps.b[1] : &maps.b[0], q_base * GPS, rt * 16, fb);
          }
        }
        if (!FASTMETA) {
          const uint16_t *sp = mat ? a.s[1] : a.s[0];
          const uint16_t *bp = mat ? a.b[1] : a.b[0];
          // runs of 4 metadata values: (row, span, run) per lane, GPS / 4 runs per span
          constexpr int RUNS = GPS / 4;
          for (int e = lane; e < 16 * QS * RUNS * (has_b ? 2 : 1); e += 32) {
            const int r = e & 15, c = (e >> 4) % RUNS, qs = (e >> 4) / RUNS % QS, isb = (e >> 4) / RUNS / QS;
            const int64_t row = (int64_t)rt * 16 + r;
            const int s = q_lo + qs;
            const int g0 = s * GPS + 4 * c;
            const uint16_t *src = (isb ? bp : sp) + row * GM + g0;
            uint32_t h[4];
  #pragma unroll
            for (int u = 0; u < 4; ++u) h[u] = (row < N && g0 + u < GM) ? (uint32_t)__ldg(src + u) : 0u;
            asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(mdst + isb * 16 * MROW + r * MROW +
                                                                ((s - q_base) * GPS + 4 * c) * 2),
                         "r"(h[0] | (h[1] << 16)), "r"(h[2] | (h[3] << 16))
                         : "memory");
          }
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(fb) : "memory");
        }
      }
      __syncwarp();
      ++j;
      if (++slot == (uint32_t)RING) {
        slot = 0;
        ph ^= 1u;
      }
    };
    for (int r = 0, rb = v_lo; rb < v_hi; ++r, rb += TR) {
      // this round's tiles and the next round's first RING: their slots were
      // last used by tiles of this round or earlier, which the consumers
      // finish before the round's barriers
      const int target = min(nv, (r + 1) * TR + RING);
      while (j < target) issue_next();
      if (KS > 1) {
        cluster.sync();
        cluster_sync_relaxed();
      }
    }
    return;
  }

  // ================= consumers =================
  // VAR 0: fp16 metadata, bf16 in and out, all compiled in; 1: the metadata
  // type of each matrix read at run time, bf16 in and out; 2: metadata type
  // and the dtypes of x and y all read at run time
  const int xdt = VAR == 2 ? a.xdt : (int)Q1_BF16, ydt = VAR == 2 ? a.ydt : (int)Q1_BF16;
  const int qi = warp % NWM, ri = warp / NWM;
  const bool active = qi < NW;
  const int span = q_lo + qi;  // groups 4 span .. 4 span + 3
  // the extra group of the first 4 (QS - NW) K-warps: group xu of span xspan
  const bool has_ex = active && qi < 4 * (QS - NW);
  const int xspan = q_lo + NW + (qi >> 2), xu = qi & 3;
  const int nthreads = NC * 32;

  // x may be the output of the preceding kernel: wait for it before reading
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // The rest is compiled twice, for warps of 4 groups and of 5 (the body is
  // the same; only the loops over the warp's groups get longer).
  auto consume = [&](auto ex) {
  constexpr int NG = decltype(ex)::value ? kQuad + 1 : kQuad;  // groups of this warp

  // ---- activation fragments of this warp's groups (token gid, word t of each
  //      group) and the per-group accumulator seeds: all loads first, then
  //      the fragments, then the groups' C/E chains interleaved
  uint32_t bfr[NG][16];
  float seed[NG][4];
  float sx[NG][2];
  // the small-group mapping's lane constants: bit pairs q0 = 2t, q1 = 2t + 1
  // of each half of a word, their masks, 1/d, and the C/E chains' a and d/2
  [[maybe_unused]] const uint32_t m0 = 0x00010001u << (2 * t), m1 = 0x00010001u << (2 * t + 1);
  const uint32_t seeds_s = smem_u32(smem + L.seeds) + (uint32_t)(warp * kMaxUnits * GPU * 64 + 16 * t);
  if (active && GW < 4) {
    const uint32_t id0 = inv_d_bits(2 * t), id1 = inv_d_bits(2 * t + 1);
    // word w, half j of unit u: lanes take k = 8j + 2t (+1) and k + 16 (+1)
    uint32_t xl[NG][8], xh[NG][8];
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      const int g = u < kQuad ? span * kQuad + u : xspan * kQuad + xu;
      const bool ok = gid < M && g < G;
#pragma unroll
      for (int wj = 0; wj < 8; ++wj) {
        const size_t k = (size_t)gid * K + (size_t)g * 128 + 32 * (wj >> 1) + 8 * (wj & 1) + 2 * t;
        xl[u][wj] = ok ? x_pair(a.x, xdt, k) : 0u;
        xh[u][wj] = ok ? x_pair(a.x, xdt, k + 16) : 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < NG; ++u)
#pragma unroll
      for (int wj = 0; wj < 8; ++wj) {
        bfr[u][2 * wj] = bmul2(prmt(xl[u][wj], xh[u][wj], 0x5410u), id0);
        bfr[u][2 * wj + 1] = bmul2(prmt(xl[u][wj], xh[u][wj], 0x7632u), id1);
      }
    // per group: rows 0..7 give C_g = sum a_q x', rows 8..15 Sx_g / 2
    const uint32_t ac0 = a_bits(2 * t), hc0 = halfd_bits(2 * t), ac1 = a_bits(2 * t + 1), hc1 = halfd_bits(2 * t + 1);
#pragma unroll
    for (int gi = 0; gi < GPU; ++gi) {
      float d[NG][4];
#pragma unroll
      for (int u = 0; u < NG; ++u) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#pragma unroll
      for (int wj = 2 * GW * gi; wj < 2 * GW * (gi + 1); ++wj)
#pragma unroll
        for (int u = 0; u < NG; ++u) mma_acc(d[u], ac0, hc0, ac1, hc1, bfr[u][2 * wj], bfr[u][2 * wj + 1]);
      if (gid == 0) {
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          const float e0 = AFFINE ? d[u][0] : d[u][0] + d[u][2], e1 = AFFINE ? d[u][1] : d[u][1] + d[u][3];
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(seeds_s + (uint32_t)((u * GPU + gi) * 64)),
                       "f"(-e0), "f"(-e1), "f"(2.f * d[u][2]), "f"(2.f * d[u][3])
                       : "memory");
        }
      }
    }
    __syncwarp();
  }
  if (active && GW == 4) {
    uint32_t xv[NG][16];
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      const int g = u < kQuad ? span * kQuad + u : xspan * kQuad + xu;
      if (gid < M && g < G) {
        // this lane's 32 activations of the group as 16 bf16 pairs; fp16 and
        // fp32 activations are rounded to bf16 (the MMA operand type) once here
        const size_t e0 = (size_t)gid * K + (size_t)g * 128 + 32 * t;
        if (xdt == Q1_F32) {
          const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const float *>(a.x) + e0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 v = __ldg(src + q);
            xv[u][2 * q] = pack_bf16x2(__uint_as_float(v.x), __uint_as_float(v.y));
            xv[u][2 * q + 1] = pack_bf16x2(__uint_as_float(v.z), __uint_as_float(v.w));
          }
        } else {
          const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.x) + e0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(src + q);
            xv[u][4 * q] = v.x; xv[u][4 * q + 1] = v.y; xv[u][4 * q + 2] = v.z; xv[u][4 * q + 3] = v.w;
          }
          if (xdt == Q1_F16) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&xv[u][q]));
              xv[u][q] = pack_bf16x2(f.x, f.y);
            }
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) xv[u][q] = 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < NG; ++u) {
#define Q1_PAIR(P) \
  bfr[u][P] = bmul2(prmt(xv[u][(P) >> 1], xv[u][8 + ((P) >> 1)], ((P) & 1) ? 0x7632u : 0x5410u), inv_d_bits(P));
      Q1_PAIR(0) Q1_PAIR(1) Q1_PAIR(2) Q1_PAIR(3) Q1_PAIR(4) Q1_PAIR(5) Q1_PAIR(6) Q1_PAIR(7)
      Q1_PAIR(8) Q1_PAIR(9) Q1_PAIR(10) Q1_PAIR(11) Q1_PAIR(12) Q1_PAIR(13) Q1_PAIR(14) Q1_PAIR(15)
#undef Q1_PAIR
    }
    // rows 0..7: C_g = sum a_p x'; rows 8..15: Sx_g / 2 = sum (d_p / 2) x'
    float d[NG][4];
#pragma unroll
    for (int u = 0; u < NG; ++u) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#define Q1_CE(JJ)                                                                                           \
  _Pragma("unroll") for (int u = 0; u < NG; ++u)                                                            \
      mma_acc(d[u], a_bits(2 * (JJ)), halfd_bits(2 * (JJ)), a_bits(2 * (JJ) + 1), halfd_bits(2 * (JJ) + 1), \
              bfr[u][2 * (JJ)], bfr[u][2 * (JJ) + 1]);
    Q1_CE(0) Q1_CE(1) Q1_CE(2) Q1_CE(3) Q1_CE(4) Q1_CE(5) Q1_CE(6) Q1_CE(7)
#undef Q1_CE
#pragma unroll
    for (int u = 0; u < NG; ++u) {
      // tokens 2t, 2t+1
      const float e0 = AFFINE ? d[u][0] : d[u][0] + d[u][2], e1 = AFFINE ? d[u][1] : d[u][1] + d[u][3];
      seed[u][0] = -e0; seed[u][1] = -e1; seed[u][2] = -e0; seed[u][3] = -e1;
      sx[u][0] = 2.f * d[u][2];
      sx[u][1] = 2.f * d[u][3];
    }
  }

  // bf16x2 (1.0, 1.0), kept in one register for every unpack LOP3 (opaque to
  // the compiler, so that it is not re-materialised per instruction)
  uint32_t kbase;
  asm volatile("mov.b32 %0, 0x3F803F80;" : "=r"(kbase));
  // word offsets of the four groups of a tile under the 64-byte swizzle (rows
  // gid and gid + 8 share it: ((r >> 1) & 3) is the same for both)
  const int swz = (gid >> 1) & 3;
  const uint32_t wlane = ring_s + qi * kTileBytes + gid * 64 + 4 * t;
  const uint32_t mlane = meta_s + gid * MROW + (GW == 4 ? (span - q_base) * 8 : 0);
  // the extra group's words and metadata, relative to those of the span
  const uint32_t xw = (uint32_t)((xspan - span) * kTileBytes + ((xu ^ swz) << 4));
  [[maybe_unused]] const uint32_t xm = (uint32_t)((xspan - span) * 8 + 2 * xu);

  // this lane's partial sums (rows gid, gid + 8 of K-warp qi; tokens 2t, 2t+1)
  const uint32_t plane = smem_u32(part) + (uint32_t)(((qi * 16 + gid) * MST + 2 * t) * 4);
  const bool pstore = 2 * t < MST;
  const uint32_t SW = (uint32_t)a.slot_words, SM = (uint32_t)a.slot_meta, PT = (uint32_t)a.part_tile;

  for (int rb = v_lo; rb < v_hi; rb += TR) {
    const int trc = min(TR, v_hi - rb);
    if (active && ri < trc) {
      // ring position of this warp's first tile of the round; from there the
      // slot pointers advance by R slots per tile
      const int j0 = rb - v_lo + ri;
      uint32_t slot = (uint32_t)(j0 % RING), ph = (uint32_t)((j0 / RING) & 1);
      uint32_t tb = wlane + slot * SW, mb = mlane + slot * SM, fb = full_s + 8 * slot;
      uint32_t pp = plane + (uint32_t)ri * PT;
      for (int lt = ri; lt < trc; lt += R) {
        // a wait that ran out has set the device error word; the results of
        // this call are then undefined, but the CTA still reaches its barriers
        mbar_wait(fb, ph);
        float acc[4];
        const bool mbf_t = VAR >= 1 && ((a.meta_bf16 >> ((NMAT == 2 && ((rb + lt) & 1)) ? 1 : 0)) & 1) != 0;
        [[maybe_unused]] const bool has_b_t = AFFINE && ((NMAT == 2 && ((rb + lt) & 1)) ? a.b[1] : a.b[0]) != nullptr;
        if constexpr (GW < 4) {
          // the lane's row base (all four words of a unit) and metadata row
          const uint32_t tq = tb - 4 * t;
#pragma unroll
          for (int gi = 0; gi < GPU; ++gi) {
            float4 sd[NG];
#pragma unroll
            for (int u = 0; u < NG; ++u) sd[u] = lds128f(seeds_s + (uint32_t)((u * GPU + gi) * 64));
            float d[NG][4];
#pragma unroll
            for (int w = GW * gi; w < GW * (gi + 1); ++w) {
              uint32_t wa[NG], wb[NG];
#pragma unroll
              for (int u = 0; u < NG; ++u) {
                const uint32_t o = (u < kQuad ? (uint32_t)((u ^ swz) << 4) : xw) + 4 * w;
                wa[u] = lds32(tq + o);
                wb[u] = lds32(tq + o + 8 * 64);
              }
#pragma unroll
              for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int u = 0; u < NG; ++u) {
                  const uint32_t ra = j ? __umulhi(wa[u], 0x01000000u) : wa[u];
                  const uint32_t rb2 = j ? __umulhi(wb[u], 0x01000000u) : wb[u];
                  const uint32_t A0 = selr(ra, m0, kbase), A1 = selr(rb2, m0, kbase);
                  const uint32_t A2 = selr(ra, m1, kbase), A3 = selr(rb2, m1, kbase);
                  if (w == GW * gi && j == 0) {
                    const float c[4] = {sd[u].x, sd[u].y, sd[u].x, sd[u].y};
                    mma_from(d[u], A0, A1, A2, A3, bfr[u][4 * w + 2 * j], bfr[u][4 * w + 2 * j + 1], c);
                  } else {
                    mma_acc(d[u], A0, A1, A2, A3, bfr[u][4 * w + 2 * j], bfr[u][4 * w + 2 * j + 1]);
                  }
                }
              }
            }
            // the group's epilogue in every unit
#pragma unroll
            for (int u = 0; u < NG; ++u) {
              const int mi = (u < kQuad ? (span - q_base) * GPS + u * GPU : (xspan - q_base) * GPS + xu * GPU) + gi;
              const float s_a = meta_f32(lds16(mb + 2 * mi), mbf_t), s_b = meta_f32(lds16(mb + 8 * MROW + 2 * mi), mbf_t);
              if (gi == 0 && u == 0) {
                acc[0] = s_a * d[u][0]; acc[1] = s_a * d[u][1]; acc[2] = s_b * d[u][2]; acc[3] = s_b * d[u][3];
              } else {
                acc[0] = fmaf(s_a, d[u][0], acc[0]); acc[1] = fmaf(s_a, d[u][1], acc[1]);
                acc[2] = fmaf(s_b, d[u][2], acc[2]); acc[3] = fmaf(s_b, d[u][3], acc[3]);
              }
              if (AFFINE) {
                float b_a, b_b;
                if (has_b_t) {
                  b_a = meta_f32(lds16(mb + 16 * MROW + 2 * mi), mbf_t);
                  b_b = meta_f32(lds16(mb + 24 * MROW + 2 * mi), mbf_t);
                } else {
                  b_a = __fmul_rn(-0.5f, s_a);
                  b_b = __fmul_rn(-0.5f, s_b);
                }
                acc[0] = fmaf(b_a, sd[u].z, acc[0]); acc[1] = fmaf(b_a, sd[u].w, acc[1]);
                acc[2] = fmaf(b_b, sd[u].z, acc[2]); acc[3] = fmaf(b_b, sd[u].w, acc[3]);
              }
            }
          }
        } else {
        uint32_t wa[NG], wb[NG];
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          const uint32_t o = u < kQuad ? (uint32_t)((u ^ swz) << 4) : xw;
          wa[u] = lds32(tb + o);
          wb[u] = lds32(tb + o + 8 * 64);
        }
        const uint2 sa = lds64(mb), sb = lds64(mb + 8 * MROW);
        uint32_t xsa = 0u, xsb = 0u, xba = 0u, xbb = 0u;
        if (NG > kQuad) {
          xsa = lds16(mb + xm);
          xsb = lds16(mb + xm + 8 * MROW);
        }
        uint2 ba = make_uint2(0, 0), bb = make_uint2(0, 0);
        const bool has_b = AFFINE && ((NMAT == 2 && ((rb + lt) & 1)) ? a.b[1] : a.b[0]) != nullptr;
        if (AFFINE && has_b) {
          ba = lds64(mb + 16 * MROW);
          bb = lds64(mb + 24 * MROW);
          if (NG > kQuad) {
            xba = lds16(mb + xm + 16 * MROW);
            xbb = lds16(mb + xm + 24 * MROW);
          }
        }
        // the words shifted right by 8, as the high half of a multiply by 2^24:
        // a multiply-add pipe instruction instead of an integer-pipe shift
        uint32_t wa8[NG], wb8[NG];
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          wa8[u] = __umulhi(wa[u], 0x01000000u);
          wb8[u] = __umulhi(wb[u], 0x01000000u);
        }
        // independent chains (one per group), interleaved step by step
        float d[NG][4];
#pragma unroll
        for (int u = 0; u < NG; ++u)
          mma_from(d[u], pair_reg<0>(wa[u], wa8[u], kbase), pair_reg<0>(wb[u], wb8[u], kbase),
                   pair_reg<1>(wa[u], wa8[u], kbase), pair_reg<1>(wb[u], wb8[u], kbase), bfr[u][0], bfr[u][1],
                   seed[u]);
#define Q1_MMA(JJ)                                                                                          \
  _Pragma("unroll") for (int u = 0; u < NG; ++u)                                                            \
      mma_acc(d[u], pair_reg<2 * (JJ)>(wa[u], wa8[u], kbase), pair_reg<2 * (JJ)>(wb[u], wb8[u], kbase),       \
              pair_reg<2 * (JJ) + 1>(wa[u], wa8[u], kbase), pair_reg<2 * (JJ) + 1>(wb[u], wb8[u], kbase),     \
              bfr[u][2 * (JJ)], bfr[u][2 * (JJ) + 1]);
        Q1_MMA(1) Q1_MMA(2) Q1_MMA(3) Q1_MMA(4) Q1_MMA(5) Q1_MMA(6) Q1_MMA(7)
#undef Q1_MMA
        const bool mbf = mbf_t;
#pragma unroll
        for (int u = 0; u < NG; ++u) {
          const float s_a = u < kQuad ? meta_half_f32(u < 2 ? sa.x : sa.y, u & 1, mbf) : meta_half_f32(xsa, 0, mbf);
          const float s_b = u < kQuad ? meta_half_f32(u < 2 ? sb.x : sb.y, u & 1, mbf) : meta_half_f32(xsb, 0, mbf);
          if (u == 0) {
            acc[0] = s_a * d[u][0]; acc[1] = s_a * d[u][1]; acc[2] = s_b * d[u][2]; acc[3] = s_b * d[u][3];
          } else {
            acc[0] = fmaf(s_a, d[u][0], acc[0]); acc[1] = fmaf(s_a, d[u][1], acc[1]);
            acc[2] = fmaf(s_b, d[u][2], acc[2]); acc[3] = fmaf(s_b, d[u][3], acc[3]);
          }
          if (AFFINE) {
            float b_a, b_b;
            if (has_b) {
              b_a = u < kQuad ? meta_half_f32(u < 2 ? ba.x : ba.y, u & 1, mbf) : meta_half_f32(xba, 0, mbf);
              b_b = u < kQuad ? meta_half_f32(u < 2 ? bb.x : bb.y, u & 1, mbf) : meta_half_f32(xbb, 0, mbf);
            } else {  // matrix without stored biases: symmetric
              b_a = __fmul_rn(-0.5f, s_a);
              b_b = __fmul_rn(-0.5f, s_b);
            }
            acc[0] = fmaf(b_a, sx[u][0], acc[0]); acc[1] = fmaf(b_a, sx[u][1], acc[1]);
            acc[2] = fmaf(b_b, sx[u][0], acc[2]); acc[3] = fmaf(b_b, sx[u][1], acc[3]);
          }
        }
        }
        // every lane's values are consumed: release the slot to the producer
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(fb + 8 * RING) : "memory");
        if (pstore) {
          asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(pp), "f"(acc[0]), "f"(acc[1]) : "memory");
          asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(pp + 8 * MST * 4), "f"(acc[2]), "f"(acc[3])
                       : "memory");
        }
        // advance R slots (the chooser keeps R < RING)
        pp += (uint32_t)R * PT;
        slot += (uint32_t)R;
        tb += (uint32_t)R * SW;
        mb += (uint32_t)R * SM;
        fb += 8u * (uint32_t)R;
        if (slot >= (uint32_t)RING) {
          slot -= (uint32_t)RING;
          tb -= (uint32_t)RING * SW;
          mb -= (uint32_t)RING * SM;
          fb -= 8u * (uint32_t)RING;
          ph ^= 1u;
        }
      }
    }
    consumer_sync(nthreads);

    // ---- combine the spans' partials of each output, in span order
    // the token index runs fastest: consecutive threads read consecutive
    // words of a partial row (no bank conflicts at M = 8)
    const int npairs = trc / NMAT;
    if (KS == 1) {
      const int cnt = npairs * 16 * M;
      for (int i = tid; i < cnt; i += nthreads) {
        const int m = i % M, r = (i / M) & 15, lp = (i / M) >> 4;
        const int lt = lp * NMAT;
        const int64_t n = (int64_t)((rb + lt) / NMAT) * 16 + r;
        // unrolled to the most K-warps a CTA holds, so that the loads need
        // not wait for the sums before them; the sums stay in K-warp order
        const float *p0 = part + ((size_t)lt * NWM * 16 + r) * MST + m;
        const float *p1 = p0 + (size_t)NWM * 16 * MST;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxWarps; ++q) {
          if (q < NW) {
            v0 += p0[(size_t)q * 16 * MST];
            if (NMAT == 2) v1 += p1[(size_t)q * 16 * MST];
          }
        }
        if (n < N) {
          const float o = NMAT == 2 ? v0 / (1.0f + expf(-v0)) * v1 : v0;  // SiLU(gate) * up
          store_act(a.out, (size_t)m * N + n, o, ydt);
        }
      }
      consumer_sync(nthreads);  // the next round rewrites the partials
    } else {
      const int cnt = trc * 16 * M;
      for (int i = tid; i < cnt; i += nthreads) {
        const int m = i % M, r = (i / M) & 15, lt = i / (16 * M);
        const float *p0 = part + ((size_t)lt * NWM * 16 + r) * MST + m;
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxWarps; ++q)
          if (q < NW) v += p0[(size_t)q * 16 * MST];
        red[((size_t)lt * 16 + r) * MST + m] = v;
      }
      cluster.sync();
      // rank k finishes 1/KS of the round's (pairs of) row tiles, summing the
      // ranks' partials in rank order
      const int per = (npairs + KS - 1) / KS;
      const int lo = min(npairs, rank * per), hi = min(npairs, lo + per);
      const int cnt2 = (hi - lo) * 16 * M;
      for (int i = tid; i < cnt2; i += nthreads) {
        const int m = i % M, r = (i / M) & 15, lp = lo + ((i / M) >> 4);
        const int lt = lp * NMAT;
        const int64_t n = (int64_t)((rb + lt) / NMAT) * 16 + r;
        // every rank's value is requested before the first one is added: the
        // remote reads overlap instead of queueing one behind the other
        const size_t o0 = ((size_t)lt * 16 + r) * MST + m, o1 = o0 + (size_t)16 * MST;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxKS; ++q) {
          if (q < KS) {
            const float *rq = cluster.map_shared_rank(red, q);
            v0 += rq[o0];
            if (NMAT == 2) v1 += rq[o1];
          }
        }
        if (n < N) {
          const float o = NMAT == 2 ? v0 / (1.0f + expf(-v0)) * v1 : v0;
          store_act(a.out, (size_t)m * N + n, o, ydt);
        }
      }
      cluster_sync_relaxed();  // every rank is done reading this round's partials
    }
  }
  };
  if (has_ex)
    consume(std::true_type{});
  else
    consume(std::false_type{});
}

// ---------------------------------------------------------------------------
// host: geometry
// ---------------------------------------------------------------------------
int sm_count_cached() {
  static std::atomic<int> cached[kMaxDevices];
  const int dev = current_device();
  if (dev < kMaxDevices && cached[dev].load(std::memory_order_relaxed) > 0)
    return cached[dev].load(std::memory_order_relaxed);
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 148;
  if (dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int NMAT, bool AFFINE, bool FASTMETA, int VAR, int GW>
int max_clusters(int ks) {
  static std::atomic<int> cache[kMaxDevices][9];
  const int dev = current_device();
  if (dev < kMaxDevices && cache[dev][ks].load(std::memory_order_relaxed) > 0)
    return cache[dev][ks].load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ks * 64), 1, 1);
  cfg.blockDim = dim3(kMaxThreads, 1, 1);
  cfg.dynamicSmemBytes = 160 * 1024;  // one CTA per SM
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)ks;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, narrow_kernel<NMAT, AFFINE, FASTMETA, VAR, GW>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = sm_count_cached() / ks;
  }
  if (n < 1) n = 1;
  if (dev < kMaxDevices) cache[dev][ks].store(n, std::memory_order_relaxed);
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
// (one span block) with the 64-byte swizzle; rows >= N and words >= K/32
// read as zero.
bool make_word_map(CUtensorMap *map, const uint32_t *w, int64_t N, int64_t K) {
  auto encode = encode_fn();
  if (!encode) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
  cuuint64_t gstride[1] = {(cuuint64_t)(K / 32) * 4};
  cuuint32_t box[2] = {16, 16};
  cuuint32_t estride[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed words [N][K/32] as a 3-D uint32 tensor (16 words of a span, rows,
// spans), boxes of 16 words x 16 rows x `spans` spans with the 64-byte
// swizzle: the smem image of one box is the per-span boxes of make_word_map
// back to back.  Only for K % 512 == 0, where every span is whole and the
// three dimensions tile each row exactly (nothing outside the array is ever
// addressed); rows >= N read as zero.
bool make_word_map3(CUtensorMap *map, const uint32_t *w, int64_t N, int64_t K, int spans) {
  auto encode = encode_fn();
  if (!encode || K % 512 != 0 || spans < 1) return false;
  cuuint64_t gdim[3] = {16, (cuuint64_t)N, (cuuint64_t)(K / 512)};
  cuuint64_t gstride[2] = {(cuuint64_t)(K / 32) * 4, 64};
  cuuint32_t box[3] = {16, 16, (cuuint32_t)spans};
  cuuint32_t estride[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t *>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scales or biases [N][G] fp16 as a 2-D uint16 tensor; boxes of box_groups
// (a multiple of 8) groups x 16 rows, no swizzle; rows >= N and groups >= G
// read as zero.  Needs G % 8 == 0 (16-byte rows) and a 16-byte aligned base.
bool make_meta_map(CUtensorMap *map, const uint16_t *m, int64_t N, int64_t G, int box_groups) {
  auto encode = encode_fn();
  if (!encode) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)G, (cuuint64_t)N};
  cuuint64_t gstride[1] = {(cuuint64_t)G * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_groups, 16};
  cuuint32_t estride[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(m), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Pick the geometry: among cluster sizes KS (K slices) whose spans fit, the
// one with the least estimated work on the busiest SM, in span-tile units:
// the group-tiles of its busiest sub-partition (a quarter of the SM's when
// balanced) or the producer's per-slot cost if that is larger, about 0.7
// tile per warp for the activation fragments, the cluster exchange, and the
// extra rounds when the partial sums do not fit at once.
template <int NMAT, bool AFFINE, bool FASTMETA, int VAR, int GW>
bool choose_geo(int64_t N, int K, int M, Geo *out) {
  const int G = K / 128;
  const int QK = (G + kQuad - 1) / kQuad;
  const int NT = (int)((N + 15) / 16);
  const int mst = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
  double best = -1.0;
  for (int ks = 1; ks <= kMaxKS; ks *= 2) {
    if (ks > QK) break;
    const int qm = (QK + ks - 1) / ks;
    if (qm > kMaxSpans) continue;
    const int nw = kwarps(qm);
    int nclus = max_clusters<NMAT, AFFINE, FASTMETA, VAR, GW>(ks);
    if (nclus > NT) nclus = NT;
    const int tv = ((NT + nclus - 1) / nclus) * NMAT;  // virtual row tiles of the widest range
    int R = kMaxWarps / nw;
    if (R > tv) R = tv;
    if (R < 1) R = 1;
    const int W = nw * R;
    // ring: row tiles in flight.  About kRingBytes of slots per SM keeps
    // enough requests in flight for this kernel, whose tile loop consumes a
    // few TB/s across the GPU; a deeper ring only lengthens the memory queues
    // that the activation loads wait in.  At least R + 1 slots, so that every
    // consumer warp can have its next tile loading.
    Geo g{ks, nclus, qm, R, tv, 2, mst};
    const SmemLayout L0 = smem_layout(g, AFFINE, GW);
    const int slot = L0.slot_words + L0.slot_meta;
    int ring = (kRingBytes + slot - 1) / slot;
    if (ring > 8) ring = 8;
    if (ring > tv) ring = tv;
    if (ring < R + 1) ring = R + 1 < tv ? R + 1 : tv;
    if (ring < 2) ring = 2;
    g.ring = ring;
    // shrink the round, then the ring, until shared memory fits
    while (smem_layout(g, AFFINE, GW).total > kSmemMax) {
      if (g.tr > 16 * NMAT) {
        g.tr = (g.tr / 2 / NMAT) * NMAT;
      } else if (g.ring > 3 && g.ring > R + 1) {
        --g.ring;
      } else if (g.tr > NMAT) {
        g.tr = (g.tr / 2 / NMAT) * NMAT;
        if (g.tr < NMAT) g.tr = NMAT;
      } else if (g.ring > 2) {
        --g.ring;
      } else {
        break;
      }
    }
    if (smem_layout(g, AFFINE, GW).total > kSmemMax) continue;
    // the producer refills a slot only after its tile is read: with R warps
    // per span, a ring shorter than R + 1 could starve a warp
    if (g.ring < (R + 1 < tv ? R + 1 : tv)) continue;
    const int rounds = (tv + g.tr - 1) / g.tr;
    // group-tiles of the busiest SM sub-partition (warp w runs on w % 4 and
    // takes its groups of every R-th row tile); qm x tv when all four carry
    // the same, more when they do not
    double load[4] = {0.0, 0.0, 0.0, 0.0};
    for (int w = 0; w < W; ++w) {
      const int q = w % nw, r = w / nw;
      const int groups = kQuad + (q < kQuad * (qm - nw) ? 1 : 0);
      load[w % 4] += (double)groups * ((tv - r + R - 1) / R);
    }
    double tiles = load[0];
    for (int i = 1; i < 4; ++i) tiles = load[i] > tiles ? load[i] : tiles;
    if (W < 8) tiles *= 1.25;  // a sub-partition with one warp hides less latency
    // the producer spends a few hundred clocks on every slot (about 3 units)
    // however small: with thin K-slices and long row ranges it sets the pace
    if (3.0 * tv > tiles) tiles = 3.0 * tv;
    const double cost = tiles + 0.7 * W + (ks > 1 ? 20.0 : 0.0) + 20.0 * (rounds - 1);
    if (best < 0 || cost < best) {
      best = cost;
      *out = g;
    }
  }
  return best >= 0;
}

template <int NMAT, bool AFFINE, bool FASTMETA, int VAR, int GW>
cudaError_t launch_impl(NarrowArgs args, const uint32_t *w0, const uint32_t *w1, cudaStream_t st, bool pdl) {
  auto kern = narrow_kernel<NMAT, AFFINE, FASTMETA, VAR, GW>;
  static std::atomic<uint64_t> attr_set{0};
  const int dev = current_device();
  if (not_done(attr_set, dev)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
    if (e != cudaSuccess) return e;
    mark_done(attr_set, dev);
  }
  Geo g;
  if (!choose_geo<NMAT, AFFINE, FASTMETA, VAR, GW>(args.N, args.K, args.M, &g)) return cudaErrorInvalidConfiguration;
  args.geo = g;
  {
    const SmemLayout L0 = smem_layout(g, AFFINE, GW);
    args.slot_words = L0.slot_words;
    args.slot_meta = L0.slot_meta;
    args.part_tile = kwarps(g.qm) * 16 * (g.mst < 2 ? 2 : g.mst) * 4;
  }
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  if (!make_word_map(&maps.w[0], w0, args.N, args.K)) return cudaErrorInvalidValue;
  if (!make_word_map(&maps.w[1], w1, args.N, args.K)) return cudaErrorInvalidValue;
  // one TMA per slot when every span is whole; a CTA holds qm or qm - 1 spans
  args.w3 = args.K % 512 == 0;
  for (int m = 0; m < 2 && args.w3; ++m)
    for (int v = 0; v < 2 && args.w3; ++v)
      if (g.qm - v >= 1 && !make_word_map3(&maps.w3[m][v], m ? w1 : w0, args.N, args.K, g.qm - v)) args.w3 = 0;
  if (FASTMETA) {
    const int64_t G = args.K / (32 * GW);
    const int box = meta_groups(g.qm, 16 / GW);
    for (int i = 0; i < 2; ++i) {
      if (!make_meta_map(&maps.s[i], args.s[i], args.N, G, box)) return cudaErrorInvalidValue;
      if (args.b[i] && !make_meta_map(&maps.b[i], args.b[i], args.N, G, box))
        return cudaErrorInvalidValue;
    }
  }
  const SmemLayout L = smem_layout(g, AFFINE, GW);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(g.nclus * g.ks), 1, 1);
  cfg.blockDim = dim3((unsigned)((kwarps(g.qm) * g.R + 1) * 32), 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = (unsigned)g.ks;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, args);
}

template <int NMAT, bool AFFINE, int VAR, int GW = 4>
cudaError_t launch_meta(NarrowArgs args, const uint32_t *w0, const uint32_t *w1, cudaStream_t st, bool pdl) {
  // metadata by TMA needs 16-byte rows (groups per row % 8 == 0) and 16-byte
  // aligned arrays
  bool fast = (args.K / (32 * GW)) % 8 == 0;
  for (int i = 0; i < 2; ++i) {
    fast = fast && (reinterpret_cast<uintptr_t>(args.s[i]) & 15) == 0;
    fast = fast && (reinterpret_cast<uintptr_t>(args.b[i]) & 15) == 0;
  }
  if (fast) return launch_impl<NMAT, AFFINE, true, VAR, GW>(args, w0, w1, st, pdl);
  return launch_impl<NMAT, AFFINE, false, VAR, GW>(args, w0, w1, st, pdl);
}

// Groups of 64 or 32 weights: one instance per group size, every type read
// at run time (VAR 2).
template <int NMAT, bool AFFINE>
cudaError_t launch_small(NarrowArgs args, const uint32_t *w0, const uint32_t *w1, int gshift, cudaStream_t st,
                         bool pdl) {
  if (gshift == 1) return launch_meta<NMAT, AFFINE, 2, 2>(args, w0, w1, st, pdl);
  return launch_meta<NMAT, AFFINE, 2, 1>(args, w0, w1, st, pdl);
}

NarrowArgs make_args(const void *x, int64_t M, int64_t N, int64_t K, void *out, q1_dtype xdt, q1_dtype ydt) {
  NarrowArgs a = {};
  a.x = x;
  a.N = N;
  a.K = (int)K;
  a.M = (int)M;
  a.out = out;
  a.xdt = (int)xdt;
  a.ydt = (int)ydt;
  return a;
}

}  // namespace

cudaError_t launch_narrow(const WeightView &W, const void *x, int64_t M, void *y,
                          cudaStream_t st, bool pdl, q1_dtype xdt, q1_dtype ydt) {
  NarrowArgs a = make_args(x, M, W.N, W.K, y, xdt, ydt);
  a.s[0] = a.s[1] = W.s;
  a.b[0] = a.b[1] = W.b;
  a.meta_bf16 = W.mbf16 ? 3 : 0;
  if (W.gshift < 2)
    return W.b ? launch_small<1, true>(a, W.w, W.w, W.gshift, st, pdl)
               : launch_small<1, false>(a, W.w, W.w, W.gshift, st, pdl);
  if (xdt != Q1_BF16 || ydt != Q1_BF16)
    return W.b ? launch_meta<1, true, 2>(a, W.w, W.w, st, pdl) : launch_meta<1, false, 2>(a, W.w, W.w, st, pdl);
  if (W.mbf16)
    return W.b ? launch_meta<1, true, 1>(a, W.w, W.w, st, pdl) : launch_meta<1, false, 1>(a, W.w, W.w, st, pdl);
  return W.b ? launch_meta<1, true, 0>(a, W.w, W.w, st, pdl) : launch_meta<1, false, 0>(a, W.w, W.w, st, pdl);
}

cudaError_t launch_narrow_gate_up(const WeightView &G, const WeightView &U, const void *x,
                                  int64_t M, void *h, cudaStream_t st, bool pdl, q1_dtype xdt) {
  NarrowArgs a = make_args(x, M, G.N, G.K, h, xdt, Q1_BF16);
  a.s[0] = G.s;
  a.s[1] = U.s;
  a.b[0] = G.b;
  a.b[1] = U.b;
  a.meta_bf16 = (G.mbf16 ? 1 : 0) | (U.mbf16 ? 2 : 0);
  // With mixed metadata the affine variant runs for both matrices; it derives
  // -scale/2 for the one whose biases pointer is null.  Gate and up share one
  // group size (the API checks it).
  if (G.gshift < 2)
    return (G.b || U.b) ? launch_small<2, true>(a, G.w, U.w, G.gshift, st, pdl)
                        : launch_small<2, false>(a, G.w, U.w, G.gshift, st, pdl);
  if (xdt != Q1_BF16) {
    if (G.b || U.b) return launch_meta<2, true, 2>(a, G.w, U.w, st, pdl);
    return launch_meta<2, false, 2>(a, G.w, U.w, st, pdl);
  }
  if (a.meta_bf16) {
    if (G.b || U.b) return launch_meta<2, true, 1>(a, G.w, U.w, st, pdl);
    return launch_meta<2, false, 1>(a, G.w, U.w, st, pdl);
  }
  if (G.b || U.b) return launch_meta<2, true, 0>(a, G.w, U.w, st, pdl);
  return launch_meta<2, false, 0>(a, G.w, U.w, st, pdl);
}

cudaError_t set_narrow_diagnostics(unsigned long long wait_ns, int stall) {
  cudaError_t e = cudaMemcpyToSymbol(c_narrow_wait_ns, &wait_ns, sizeof(wait_ns));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(c_narrow_stall, &stall, sizeof(stall));
  return e;
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
