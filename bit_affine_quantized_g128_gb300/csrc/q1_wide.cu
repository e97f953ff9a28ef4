// Wide (prefill) Q1 matmul on the tcgen05 tensor cores:
//   y[M][N] = x[M][K] . Wd^T, fp32 accumulation in tensor memory.
//
// The page "Support Bonsai-27B affine Q1" (higgs PR #212), section
// "Limitations / non-goals", runs forwards wider than the narrow threshold by
// dequantizing the whole matrix to the input dtype and calling a dense matmul,
// which is what set its peak memory ("Measured impact": peak about 6.65 GB
// from dense prefill temporaries).  Here the dequantization happens per stage
// straight into tensor memory, feeding the MMA: no dense weight temporary.
//
// Operand precision.  Rounding the dequantized weights to bf16 (a half-ulp of
// 2^-8, the same for every weight of a symmetric group) moves a few outputs in
// 10^5 past the per-element error bar the method is held to, so the operands
// are fp16 instead: symmetric weights +-s/2 are exact in fp16 and affine
// values s+b are rounded once at 2^-11.  The activations go to fp16 through a
// per-row power-of-two scale 2^e_m chosen so that the row maximum lands in
// [2^14, 2^15) (exact for every normal fp16 result, no overflow); the
// epilogue multiplies by 2^-e_m.  A small prep kernel writes the scaled fp16
// rows and the scales into the caller's workspace.
//
// The matmul runs on CTA pairs (tcgen05.mma.cta_group::2): the pair computes
// 256 weight rows x NT tokens, the dequantized weights are the MMA's A
// operand in tensor memory (M = 256, 128 rows per CTA) and the activations
// the B operand in shared memory (N = NT, NT/2 tokens per CTA), K = 16 per
// instruction.  Weights written to tensor memory by tcgen05.st never touch
// shared memory, and each CTA holds only its half of the token tile, so
// shared memory carries about 64 B/clk at full MMA rate.  (With the weights
// as the shared-memory operand instead, every MMA re-read the weight tile
// from shared memory and the dequantizers' stores drained slowly behind those
// reads: the k-steps ran at about half the MMA rate.)
#include <type_traits>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace q1 {

__device__ unsigned int g_wide_err = 0;
// Diagnostics (set from the host between launches): the limit of every
// bounded wait, and a switch that makes the x producer issue nothing, so that
// every wait for its data runs out (no copy is then in flight).
__constant__ unsigned long long c_wide_wait_ns = 2000000000ull;
__constant__ int c_wide_stall = 0;

namespace {



__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
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

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), fixed
// descriptor version 1 at bits 46..48, swizzle mode 2 (128B) at bits 61..63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
  d |= (uint64_t)1 << 46;             // version
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 32 weights of one word -> 16 pairs of 16-bit values in k order: out[j] =
// (k = 2j, 2j+1), each lo (bit 0) or hi (bit 1) of the group.
// A prmt with the sign-replicate selector turns bit 7 of a source byte into a
// 0x00/0xFF byte, so two shifted copies of the word give 16-bit masks for two
// adjacent weights at once; one LOP3 then selects hi (bit 1) or lo (bit 0).
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t lo2, uint32_t hi2, uint32_t (&out)[16]) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const uint32_t A = w << (7 - e);  // byte i msb = bit 8i+e
    const uint32_t B = w << (6 - e);  // byte i msb = bit 8i+e+1
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t s = (8u | i) | ((8u | i) << 4) | ((8u | (4 + i)) << 8) | ((8u | (4 + i)) << 12);
      const uint32_t m = prmt(A, B, s);
      out[4 * i + e / 2] = (m & hi2) | (~m & lo2);
    }
  }
}

// Output stores in the activation dtype, one rounding for 16-bit types.
__device__ __forceinline__ void store1(void *y, size_t i, float v, int dt) {
  if (dt == Q1_F32) static_cast<float *>(y)[i] = v;
  else if (dt == Q1_F16) static_cast<__half *>(y)[i] = __float2half_rn(v);
  else static_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, int dt) {
  if (dt == Q1_F16) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
  }
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// four values, y + i aligned to 8 bytes (16-bit types) or 16 bytes (fp32)
__device__ __forceinline__ void store4(void *y, size_t i, const float (&f)[4], int dt) {
  if (dt == Q1_F32) {
    *reinterpret_cast<float4 *>(static_cast<float *>(y) + i) = make_float4(f[0], f[1], f[2], f[3]);
  } else {
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(y) + i) = make_uint2(pack2(f[0], f[1], dt), pack2(f[2], f[3], dt));
  }
}

// x [M][K] bf16 -> x16 [M][K] fp16 = x * 2^e_m and inv_scale[m] = 2^-e_m, with
// Eight activations x[m][8i .. 8i+7] as fp32 (bf16 and fp16 widen exactly).
template <int XDT>
__device__ __forceinline__ void load8(const void *__restrict__ row, int i, float (&f)[8]) {
  if (XDT == Q1_F32) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row) + 2 * i;
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(w[j]);
  } else {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (XDT == Q1_F16) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[q]));
        f[2 * q] = t.x;
        f[2 * q + 1] = t.y;
      } else {
        f[2 * q] = __uint_as_float(w[q] << 16);
        f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
  }
}

// e_m = 14 - floor(log2(max_k |x[m][k]|)) so that the row maximum lands in
// [2^14, 2^15).  Multiplying by a power of two is exact; the fp16 rounding is
// exact for every bf16 or fp16 activation whose scaled value is a normal fp16
// number, and rounds fp32 activations once (2^-11).  One block of 256 threads
// per row.  Rows of at most kPrepHeld chunks of 8 per thread are read once:
// each thread keeps its chunks in registers between the maximum and the
// conversion.  Longer rows take two passes: the maximum pass keeps four
// independent loads in flight per thread, and the conversion pass reads the
// row again (mostly from L2).
constexpr int kPrepThreads = 256;
constexpr int kPrepHeld = 4;
template <int XDT, bool HELD>
__global__ void __launch_bounds__(kPrepThreads) x_to_f16_kernel(const void *__restrict__ x, int K,
                                                                __half *__restrict__ x16,
                                                                float *__restrict__ inv_scale,
                                                                int *__restrict__ cnt, int ncnt) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the stream schedule's share counts start at zero
  for (int i = blockIdx.x * kPrepThreads + threadIdx.x; i < ncnt; i += gridDim.x * kPrepThreads) cnt[i] = 0;
  __shared__ float wmax[kPrepThreads / 32];
  const int m = blockIdx.x, tid = threadIdx.x;
  const void *row = static_cast<const char *>(x) + (size_t)m * K * (XDT == Q1_F32 ? 4 : 2);
  const int n8 = K / 8;  // chunks of 8 activations
  float mx = 0.f;
  float fh[HELD ? kPrepHeld : 1][8];  // the held chunks tid + u * kPrepThreads
  if constexpr (HELD) {
#pragma unroll
    for (int u = 0; u < kPrepHeld; ++u) {
      const int c = tid + u * kPrepThreads;
      if (c < n8) {
        load8<XDT>(row, c, fh[u]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) fh[u][j] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kPrepHeld; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(fh[u][j]));
  }
  int i = HELD ? n8 : tid;
  for (; i + 3 * kPrepThreads < n8; i += 4 * kPrepThreads) {
    float f[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) load8<XDT>(row, i + u * kPrepThreads, f[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[u][j]));
  }
  for (; i < n8; i += kPrepThreads) {
    float f[8];
    load8<XDT>(row, i, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) wmax[tid >> 5] = mx;
  __syncthreads();
  mx = wmax[0];
#pragma unroll
  for (int w = 1; w < kPrepThreads / 32; ++w) mx = fmaxf(mx, wmax[w]);
  int e = 0;
  if (mx > 0.f && mx <= 3.0e38f) {
    const int E = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2) for normal mx
    e = 14 - (E < -126 ? -126 : E);
    if (e > 126) e = 126;
    if (e < -126) e = -126;
  }
  const float sc = __uint_as_float((uint32_t)(127 + e) << 23);   // 2^e, exact
  const float isc = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, exact
  uint4 *out = reinterpret_cast<uint4 *>(x16 + (size_t)m * K);
  auto convert = [&](const float (&f)[8], int c) {
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(f[2 * q] * sc, f[2 * q + 1] * sc);
      o[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    out[c] = make_uint4(o[0], o[1], o[2], o[3]);
  };
  if constexpr (HELD) {
#pragma unroll
    for (int u = 0; u < kPrepHeld; ++u) {
      const int c = tid + u * kPrepThreads;
      if (c < n8) convert(fh[u], c);
    }
  } else {
#pragma unroll 4
    for (int c = tid; c < n8; c += kPrepThreads) {
      float f[8];
      load8<XDT>(row, c, f);
      convert(f, c);
    }
  }
  if (tid == 0) inv_scale[m] = isc;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// ======================================================================
// Pair kernel.  Per CTA (576 threads), CTA h of the pair owning weight rows
// n0 + 128h .. n0 + 128h + 127 of the tile:
//   warp 0        TMA producer: this CTA's NT/2 tokens x 128 k of fp16 x per
//                 stage (two 128B-swizzled boxes of 64 k), up to 8 stages ahead
//   warp 1        TMEM allocation for the pair (512 columns: the fp32
//                 accumulator in columns [0, 256), four 64-column weight
//                 stages in [256, 512)); in the even CTA one thread issues the
//                 pair's MMAs and commits them to both CTAs' barriers
//   warps 2..9    dequantizers, two sets of four taking alternate stages:
//                 thread = weight row, four words (128 k) -> 64 fp16 pairs ->
//                 tcgen05.st; then, once this CTA's x stage has landed, one
//                 arrival per warp on the even CTA's stage barrier
//   warps 10..17  epilogue: tcgen05.ld -> x 2^-e_m per token -> output dtype
//                 -> a staged tile and one TMA store per tile (16-bit outputs)
//                 or direct stores (a warp's store covers 32 consecutive rows)
// Tiles (256 weight rows x NT tokens) are taken persistently by the pairs;
// the accumulator is released to the next tile as soon as it has been read.
// With SPLIT, a cluster of S pairs shares one tile, pair p taking the p-th of
// S contiguous k ranges, and the fp32 partial tiles are summed through
// distributed shared memory in pair order (deterministic).
constexpr int kPairThreads = 576;
// TMEM (512 columns): the fp32 accumulator of a tile takes NT columns, a
// 128-k weight stage 64.  Token tiles up to 160 get two accumulators
// ([0, NT) and [160, 160 + NT)) and three weight stages in [320, 512): the
// epilogue of one tile then runs under the next tile's MMAs.  Wider tiles get
// one accumulator in [0, 256) and four weight stages in [256, 512).
constexpr int kPairAStages = 4;              // at most 4 weight stages
constexpr int kPairDbufMaxNT = 160;          // widest token tile with two accumulators
constexpr int kPairXMax = 8;                 // at most 8 x stages of 128 k in shared memory
constexpr uint32_t kPairDeqWarp0 = 2, kPairEpiWarp0 = 10;
// Dynamic shared memory, in this order (every part 1024-byte aligned):
//   the barriers (one 1024-byte header),
//   the x ring: xstages x (NT/2 tokens x 128 k fp16), as many stages as fit;
//     after the k loop of a split-K tile it holds the fp32 partial tile,
//     token-major [NT][128] (a warp's accesses cover 32 consecutive weight rows)
//   the 16-bit output tile [NT][128] of this CTA's rows, staged for one TMA store.
constexpr size_t kPairSmemMax = 232448;      // the per-block opt-in limit
constexpr size_t kPairHeader = 1024;

struct __align__(8) PairShared {
  uint64_t full_x[kPairXMax];     // this CTA's x stage landed (TMA bytes)
  uint64_t empty_x[kPairXMax];    // the pair's MMAs reading the x stage completed (commit, both CTAs)
  uint64_t full[kPairAStages];    // even CTA: both CTAs' weights + x of the step ready (8 warps)
  uint64_t empty[kPairAStages];   // the pair's MMAs reading the weight stage completed (commit, both CTAs)
  uint64_t accum_full[2];         // the tile's MMAs completed (commit, both CTAs), per accumulator
  uint64_t accum_empty[2];        // even CTA: both CTAs' epilogues loaded the accumulator (16 warps)
  uint64_t drain;                 // final commit before the allocation is released
  uint64_t stg_ready;             // the epilogue warps' rows of the output tile are staged (8 warps)
  uint64_t stg_free;              // the previous tile's TMA store has read the staging buffer
  uint64_t part_done;             // stream: the epilogue warps' partial sums are written (8 warps)
  uint64_t last_ready;            // stream: the share's count is taken and last_flag set
  volatile int last_flag;         // stream: this CTA completed the tile's shares
  uint32_t tmem_base;
  volatile int abort_flag;
};
static_assert(sizeof(PairShared) <= kPairHeader, "barrier header");
// x stages that fit beside the staging tile for a token tile of NT (at least 4:
// the split-K partial tile, NT x 128 fp32, lives in the ring)
__host__ __device__ constexpr int pair_xstages(int NT) {
  return (int)((kPairSmemMax - 1024 - kPairHeader - (size_t)NT * 256) / ((size_t)NT * 128)) < kPairXMax
             ? (int)((kPairSmemMax - 1024 - kPairHeader - (size_t)NT * 256) / ((size_t)NT * 128))
             : kPairXMax;
}
__host__ __device__ constexpr size_t pair_smem_bytes(int NT) {
  return 1024 + kPairHeader + (size_t)pair_xstages(NT) * NT * 128 + (size_t)NT * 256;
}
static_assert(pair_xstages(256) >= 4 && pair_smem_bytes(256) <= kPairSmemMax, "pair kernel shared memory");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the same shared-memory offset in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t mapa_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA of the cluster (default semantics:
// release at CTA scope).  What the arrival publishes is complete before it:
// tensor-memory stores are waited for (tcgen05.wait::st) and fenced, and x
// stages were observed complete on their own barrier.  A cluster-scope
// release measured about 1000 clocks more per arrival, on the critical path.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bounded wait, slow path: polls the phase with the given parity until it has
// completed, the limit runs out, or any CTA has recorded an error (the pair's
// roles depend on each other's progress).  `sleep` spaces the polls of long
// waits (the epilogue's) so that they take few issue slots from the
// dequantizers.
__device__ __noinline__ bool pair_wait_slow(uint32_t addr, uint32_t parity, PairShared *sh, int sleep) {
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (sleep) __nanosleep(sleep);
    if (mbar_try(addr, parity)) return true;
    if ((i & 15u) == 15u) {
      if (sh->abort_flag || *(volatile unsigned int *)&g_wide_err) {
        sh->abort_flag = 1;
        return false;
      }
      if (globaltimer() - t0 > c_wide_wait_ns) {
        sh->abort_flag = 1;
        atomicOr(&g_wide_err, 1u);
        return false;
      }
    }
  }
}
// one thread: an inline test first, the polling loop only when the phase is open
__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, PairShared *sh, int sleep) {
  const uint32_t addr = smem_u32(bar);
  return mbar_try(addr, parity) || pair_wait_slow(addr, parity, sh, sleep);
}
// a whole warp: every lane tests once (no divergence when the phase has
// completed); otherwise lane 0 polls and the warp takes its verdict
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, PairShared *sh, int sleep) {
  const uint32_t addr = smem_u32(bar);
  if (__all_sync(0xffffffffu, mbar_try(addr, parity))) return true;
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = pair_wait_slow(addr, parity, sh, sleep);
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrives on the barrier at this offset in both CTAs of the pair once every
// MMA issued so far by this thread has completed
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// 32 columns of this warp's 32 lanes; tcgen05.wait::ld before the values are used
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
        "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
        "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  tmem_ld32_issue(taddr, v);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 2-D tiled store from shared memory (bulk-group completion)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}

// fp16x2 patterns of a group's two dequantized values (q = 0, q = 1): the
// fp32 metadata result rounded once to fp16
__device__ __forceinline__ void deq_pair(uint32_t s16, uint32_t b16, bool affine, bool mbf16, uint32_t &lo2,
                                         uint32_t &hi2) {
  const float sc = meta_f32(s16, mbf16);
  const float bi = affine ? meta_f32(b16, mbf16) : __fmul_rn(-0.5f, sc);
  const uint32_t lo16 = __half_as_ushort(__float2half_rn(bi));
  const uint32_t hi16 = __half_as_ushort(__float2half_rn(__fadd_rn(sc, bi)));
  lo2 = lo16 | (lo16 << 16);
  hi2 = hi16 | (hi16 << 16);
}

// A pair's work as segments: tile t with k-steps [ka, kb).  Round robin:
// whole tiles t, t + t_step, ... (k-steps [lo, hi) of a split).  Stream:
// the contiguous units [u, u1) of the flattened (tile, k-step) space, so
// that a tile at either end of the range may be shared with the neighbour
// pairs.
struct SegIter {
  int stream, T, KS, t, t_step, lo, hi, u, u1;
  __device__ __forceinline__ bool next(int &tt, int &ka, int &kb) {
    if (stream) {
      if (u >= u1) return false;
      tt = u / KS;
      ka = u - tt * KS;
      kb = min(KS, ka + (u1 - u));
      u += kb - ka;
      return true;
    }
    if (t >= T) return false;
    tt = t;
    ka = lo;
    kb = hi;
    t += t_step;
    return true;
  }
};

// One 128-k stage of one weight row: four words and their metadata.
struct PairStage {
  uint4 w;
  uint32_t s[4], b[4];
};

template <bool SPLIT, bool G128>
__global__ void __launch_bounds__(kPairThreads, 1)
pair_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_y,
            const uint32_t *__restrict__ W, const uint16_t *__restrict__ S, const uint16_t *__restrict__ Bv,
            int M, int N, int K, const float *__restrict__ inv_scale, void *__restrict__ y, int NT, int ksplit,
            int mbf16, int ydt, int gshift, int ystage, int stream, float *__restrict__ part,
            int *__restrict__ cnt) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  PairShared *sh = reinterpret_cast<PairShared *>(base);
  unsigned char *ring = base + kPairHeader;
  const int xstages = pair_xstages(NT);
  const uint32_t XS = (uint32_t)NT * 128u;         // bytes of one x stage (NT/2 tokens x 256 B)
  uint16_t *stg = reinterpret_cast<uint16_t *>(ring + (size_t)xstages * XS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_rank();
  const int h = (int)(crank & 1u);                 // half of the pair: weight rows 128h ..
  const uint32_t lead = crank & ~1u;               // the pair's even CTA
  const uint16_t pair_mask = (uint16_t)(3u << lead);
  const int XH = NT >> 1;                          // tokens whose x this CTA holds
  const int KS = K / 128;                          // 128-k stages of a whole row
  const int mtiles = (M + NT - 1) / NT, ntiles = (N + 255) / 256;
  // this pair's tiles and k range
  int t_first, t_step, ks_lo, ks_hi;
  if (SPLIT) {
    const int pr = (int)(crank >> 1);              // pair within the cluster
    t_first = (int)(blockIdx.x / (unsigned)(2 * ksplit));
    t_step = 1 << 30;                              // one tile per cluster
    ks_lo = (int)(((int64_t)KS * pr) / ksplit);
    ks_hi = (int)(((int64_t)KS * (pr + 1)) / ksplit);
  } else {
    t_first = (int)(blockIdx.x >> 1);
    t_step = (int)(gridDim.x >> 1);
    ks_lo = 0;
    ks_hi = KS;
  }
  const int T = mtiles * ntiles;
  const int nks = ks_hi - ks_lo;
  // stream schedule: pair pidx of P takes units [b(pidx), b(pidx + 1)), b(p) = p W / P
  const int P = (int)(gridDim.x >> 1), pidx = (int)(blockIdx.x >> 1);
  const int64_t Wu = (int64_t)T * KS;
  const int u0 = stream ? (int)((int64_t)pidx * Wu / P) : 0;
  const int u1 = stream ? (int)((int64_t)(pidx + 1) * Wu / P) : 0;
  const SegIter segs0{stream, T, KS, t_first, t_step, ks_lo, ks_hi, u0, u1};

  if (tid == 0) {
    for (int s = 0; s < xstages; ++s) {
      mbar_init(&sh->full_x[s], 1);
      mbar_init(&sh->empty_x[s], 1);
    }
    for (int s = 0; s < kPairAStages; ++s) {
      mbar_init(&sh->full[s], 8);
      mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->accum_full[b], 1);
      mbar_init(&sh->accum_empty[b], 16);
    }
    mbar_init(&sh->drain, 1);
    mbar_init(&sh->stg_ready, 8);
    mbar_init(&sh->stg_free, 1);
    mbar_init(&sh->part_done, 8);
    mbar_init(&sh->last_ready, 1);
    sh->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  cluster_sync_all();  // barriers initialised and TMEM allocated in every CTA of the cluster
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = sh->tmem_base;
  const uint32_t full_lead0 = mapa_rank(smem_u32(&sh->full[0]), lead);
  const uint32_t accum_empty_lead0 = mapa_rank(smem_u32(&sh->accum_empty[0]), lead);
  // accumulators and weight stages in TMEM (see kPairDbufMaxNT)
  const bool dbuf = !SPLIT && NT <= kPairDbufMaxNT;
  const uint32_t SA = dbuf ? 3u : 4u, a_col0 = 512u - 64u * SA, nbuf = dbuf ? 2u : 1u;

  if (warp == 0) {
    // ---------------- TMA producer: this CTA's token half, two 64-k boxes per stage
    // ((diagnostics) a stalled producer issues nothing)
    if (lane == 0 && !c_wide_stall) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // x16 comes from the prep kernel
      uint32_t s = 0, ph = 0;
      bool ok = true;
      SegIter segs = segs0;
      int t, ka, kb;
      while (ok && segs.next(t, ka, kb)) {
        const int m0 = (t % mtiles) * NT;
        for (int ks = ka; ks < kb; ++ks) {
          if (!(ok = pair_wait(&sh->empty_x[s], ph ^ 1u, sh, 0))) break;
          unsigned char *dst = ring + s * XS;
          mbar_arrive_expect_tx(&sh->full_x[s], XS);
          tma_load_2d(dst, &tmap_x, &sh->full_x[s], ks * 128, m0 + h * XH);
          tma_load_2d(dst + XS / 2, &tmap_x, &sh->full_x[s], ks * 128 + 64, m0 + h * XH);
          if (++s == (uint32_t)xstages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (even CTA)
    if (h == 0 && lane == 0) {
      const uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
      uint32_t s = 0, ph = 0, tl = 0, sx = 0;
      bool ok = true;
      SegIter segs = segs0;
      int t, ka, kb;
      for (; ok && segs.next(t, ka, kb); ++tl) {
        // accumulator b of this segment, used for the u-th time
        const uint32_t b = tl % nbuf, u = tl / nbuf, d_tmem = tmem + 160u * b;
        if (u > 0 && !(ok = pair_wait(&sh->accum_empty[b], (u - 1) & 1u, sh, 0))) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int ks = ka; ks < kb; ++ks) {
          if (!(ok = pair_wait(&sh->full[s], ph, sh, 0))) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t xs = smem_u32(ring + sx * XS);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_pair(d_tmem, tmem + a_col0 + 64u * s + 8u * kk,
                      sw128_desc(xs + (kk >> 2) * (XS / 2) + (kk & 3) * 32), idesc, (ks > ka || kk > 0) ? 1u : 0u);
          umma_commit_pair(&sh->empty[s], pair_mask);
          umma_commit_pair(&sh->empty_x[sx], pair_mask);
          if (++sx == (uint32_t)xstages) sx = 0;
          if (++s == SA) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&sh->accum_full[b], pair_mask);
      }
      umma_commit_pair(&sh->drain, pair_mask);  // every MMA issued, complete
    }
    // both CTAs see the pair's last commit arrive before the allocation is released
    if (lane == 0) pair_wait(&sh->drain, 0, sh, 0);
  } else if (warp < (int)kPairEpiWarp0) {
    // ---------------- dequantizers: set ds takes this CTA's stages it = ds (mod 2)
    const int ds = (warp - (int)kPairDeqWarp0) >> 2, q = warp & 3;
    const int r = 32 * q + lane;                   // TMEM lane = weight row of this CTA
    const int wpr = K / 32, G = wpr >> gshift;     // words and metadata groups per row
    const bool affine = Bv != nullptr, mb = mbf16 != 0;
    const uint32_t a_lane = tmem + ((uint32_t)(32 * q) << 16) + a_col0;
    // this CTA's k-steps in order: tile t, k-step ks in [lo, hi); a tile move
    // adds tstep to t and takes ks back by span (round robin: whole tiles of
    // the split's k range; stream: consecutive tiles of the unit range)
    const int my_tiles = t_first < T ? (T - 1 - t_first) / t_step + 1 : 0;
    const uint32_t total = stream ? (uint32_t)(u1 - u0) : (uint32_t)nks * (uint32_t)my_tiles;
    const int k_lo = stream ? 0 : ks_lo, k_hi = stream ? KS : ks_hi, k_span = k_hi - k_lo;
    const int k_tstep = stream ? 1 : t_step;
    // A cursor over this set's stages: tile t, k-step ks and this thread's
    // weight row n (-1 past the last tile).  It moves two stages at a time;
    // only a move to the next tile costs a division.
    struct Cursor {
      int t, ks, n;
    };
    auto set_row = [&](Cursor &c) { c.n = c.t < T ? (c.t / mtiles) * 256 + 128 * h + r : -1; };
    auto advance = [&](Cursor &c, int by) {
      c.ks += by;
      if (c.ks >= k_hi) {
        while (c.ks >= k_hi) {
          c.ks -= k_span;
          if (c.t < T) c.t += k_tstep;
        }
        set_row(c);
      }
    };
    auto load = [&](const Cursor &c, PairStage &p) {
      if (c.n >= 0 && c.n < N) {
        const int n = c.n, ks = c.ks;
        p.w = __ldg(reinterpret_cast<const uint4 *>(W + (size_t)n * wpr) + ks);
        const uint16_t *srow = S + (size_t)n * G;
        const uint16_t *brow = affine ? Bv + (size_t)n * G : nullptr;
        if (G128) {
          p.s[0] = srow[ks];
          p.b[0] = affine ? brow[ks] : 0u;
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int g = (4 * ks + u) >> gshift;
            p.s[u] = srow[g];
            p.b[u] = affine ? brow[g] : 0u;
          }
        }
      } else {
        p.w = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) p.s[u] = p.b[u] = 0u;
      }
    };
    // this set's stages j, j + 2, j + 4: the loads run two of its stages ahead
    PairStage cur, nx1, nx2;
    uint32_t j = (uint32_t)ds;
    uint32_t xj = (uint32_t)ds, xph = 0;           // x stage of step j and its phase (xstages >= 4)
    uint32_t s = (uint32_t)ds, ph = 0;             // weight stage of step j and its phase (SA >= 3)
    Cursor pf{stream ? u0 / KS : t_first, stream ? u0 % KS : ks_lo, 0};
    set_row(pf);
    advance(pf, ds);  // stage ds may already lie in the next tile
    if (j < total) load(pf, cur);
    advance(pf, 2);
    if (j + 2 < total) load(pf, nx1);
    advance(pf, 2);
    for (; j < total; j += 2) {
      if (!warp_wait(&sh->empty[s], ph ^ 1u, sh, 0)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");  // the MMAs that read the slot are done
      const uint32_t words[4] = {cur.w.x, cur.w.y, cur.w.z, cur.w.w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int u = 2 * half + u2;
          uint32_t lo2, hi2;
          deq_pair(G128 ? cur.s[0] : cur.s[u], G128 ? cur.b[0] : cur.b[u], affine, mb, lo2, hi2);
          uint32_t out[16];
          expand_word(words[u], lo2, hi2, out);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[16 * u2 + e] = out[e];
        }
        tmem_st32(a_lane + 64u * s + 32u * half, v);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // this CTA's x half of the step must have landed before the pair's MMA may run
      if (!warp_wait(&sh->full_x[xj], xph, sh, 0)) break;
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      // the even CTA's own warps signal at CTA scope; the odd CTA's at cluster
      // scope.  No load is in flight here: a cluster-scope release would wait
      // for it.
      if (lane == 0) {
        if (h == 0) mbar_arrive(&sh->full[s]);
        else mbar_arrive_remote(full_lead0 + 8u * s);
      }
      if (j + 4 < total) load(pf, nx2);
      advance(pf, 2);
      cur = nx1;
      nx1 = nx2;
      xj += 2;
      if (xj >= (uint32_t)xstages) {
        xj -= (uint32_t)xstages;
        xph ^= 1u;
      }
      s += 2;
      if (s >= SA) {
        s -= SA;
        ph ^= 1u;
      }
    }
  } else {
    // ---------------- epilogue: warp (q, eh) reads TMEM lanes 32q.. and half eh of the token columns
    const int q = warp & 3, eh = (warp - (int)kPairEpiWarp0) >> 2;
    const int r = 32 * q + lane;
    uint32_t tl = 0, ts = 0, pc = 0;  // segments, staged tiles and partial shares so far
    bool deps = false;
    SegIter segs = segs0;
    int t, ka, kb;
    // the pair holding unit v of the stream schedule, and the first unit of pair p
    auto pair_of_unit = [&](int64_t v) { return (int)(((v + 1) * P + Wu - 1) / Wu) - 1; };
    auto first_unit = [&](int p) { return (int64_t)p * Wu / P; };
    for (; segs.next(t, ka, kb); ++tl) {
      const uint32_t b = tl % nbuf, u = tl / nbuf;
      const uint32_t d_lane = tmem + ((uint32_t)(32 * q) << 16) + 160u * b;
      const uint32_t accum_empty_lead = accum_empty_lead0 + 8u * b;
      if (!warp_wait(&sh->accum_full[b], u & 1u, sh, 64)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (!deps) {
        asm volatile("griddepcontrol.wait;" ::: "memory");  // inv_scale comes from the prep kernel
        deps = true;
      }
      const int m0 = (t % mtiles) * NT;
      const int n = (t / mtiles) * 256 + 128 * h + r;
      // the two warps of a lane quarter take halves of the NT columns (multiples of 16)
      const int chalf = ((NT >> 1) + 15) & ~15;
      const int c_lo = eh * chalf, c_hi = min(NT, c_lo + chalf);
      if (stream && !(ka == 0 && kb == KS)) {
        // A share of tile t (k-steps [ka, kb)): its fp32 partial sums go to
        // this pair's workspace slot, token-major [NT][128] per CTA half; the
        // share that completes the tile's count last adds all shares in k
        // order (a fixed order: the result does not depend on which is last)
        // and writes the outputs.  No CTA waits for another.
        const int64_t tb = (int64_t)t * KS;
        const int p0 = pair_of_unit(tb), p1 = pair_of_unit(tb + KS - 1);
        const int which = (int64_t)u0 >= tb ? 0 : 1;  // this pair's first segment, or its last
        float *mine = part + ((size_t)(2 * pidx + which) * 2 + h) * ((size_t)NT * 128);
        bool released = false;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
          uint32_t va[32], vb[32];
          tmem_ld32_issue(d_lane + (uint32_t)c0, va);
          tmem_ld32_issue(d_lane + (uint32_t)(c0 + 32), vb);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (c0 + 64 >= c_hi) {
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              if (h == 0) mbar_arrive(&sh->accum_empty[b]);
              else mbar_arrive_remote(accum_empty_lead);
            }
            released = true;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < c_hi) mine[(size_t)(c0 + e) * 128 + r] = __uint_as_float(va[e]);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + 32 + e < c_hi) mine[(size_t)(c0 + 32 + e) * 128 + r] = __uint_as_float(vb[e]);
        }
        if (!released) {
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            if (h == 0) mbar_arrive(&sh->accum_empty[b]);
            else mbar_arrive_remote(accum_empty_lead);
          }
        }
        __threadfence();  // the partial sums are visible device-wide before the count
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->part_done);
        if (warp == (int)kPairEpiWarp0 && lane == 0) {
          int last = 0;
          if (pair_wait(&sh->part_done, pc & 1u, sh, 0)) {
            const int old = atomicAdd(&cnt[2 * t + h], 1);
            last = old == p1 - p0;
            if (last) cnt[2 * t + h] = 0;  // every share has counted: ready for the next call
            __threadfence();
          }
          sh->last_flag = last;
          mbar_arrive(&sh->last_ready);
        }
        if (!warp_wait(&sh->last_ready, pc & 1u, sh, 0)) break;
        ++pc;
        if (sh->last_flag) {
          __threadfence();
          // token c by warp c mod 8; lane l adds rows 4l .. 4l+3 over the shares
          const int m0 = (t % mtiles) * NT, nb = (t / mtiles) * 256 + 128 * h;
          // four tokens per round, every share's loads issued before they
          // are added (the shares sit in L2; one round trip per round)
          const int n4 = nb + 4 * lane;
          const int ctop = min(NT, M - m0);
          constexpr int kTok = 4;
          for (int c0 = (warp - (int)kPairEpiWarp0) * kTok; c0 < ctop; c0 += 8 * kTok) {
            float4 acc[kTok];
#pragma unroll
            for (int q2 = 0; q2 < kTok; ++q2) acc[q2] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = 0; i <= p1 - p0; ++i) {
              const int pi = p0 + i;
              const int wi = (i == 0 && first_unit(pi) < tb) ? 1 : 0;
              const float *src = part + ((size_t)(2 * pi + wi) * 2 + h) * ((size_t)NT * 128) + 4 * lane;
              float4 v[kTok];
#pragma unroll
              for (int q2 = 0; q2 < kTok; ++q2)
                v[q2] = c0 + q2 < ctop ? __ldcg(reinterpret_cast<const float4 *>(src + (size_t)(c0 + q2) * 128))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int q2 = 0; q2 < kTok; ++q2) {
                acc[q2].x += v[q2].x;
                acc[q2].y += v[q2].y;
                acc[q2].z += v[q2].z;
                acc[q2].w += v[q2].w;
              }
            }
            if (n4 < N) {
#pragma unroll
              for (int q2 = 0; q2 < kTok; ++q2) {
                const int m = m0 + c0 + q2;
                if (c0 + q2 < ctop) {
                  const float rs = inv_scale[m];
                  const float a4[4] = {acc[q2].x * rs, acc[q2].y * rs, acc[q2].z * rs, acc[q2].w * rs};
                  const size_t i0 = (size_t)m * N + n4;
                  if (n4 + 4 <= N && (N & 3) == 0) {
                    store4(y, i0, a4, ydt);
                  } else {
                    for (int e = 0; e < 4 && n4 + e < N; ++e) store1(y, i0 + e, a4[e], ydt);
                  }
                }
              }
            }
          }
        }
        continue;
      }
      if (!SPLIT && ystage) {
        // 16-bit outputs through the staging tile: the accumulator is released
        // as soon as it is read, and one TMA store writes the CTA's 128 rows x
        // NT tokens (clipping rows and tokens beyond N and M)
        if (ts > 0 && !warp_wait(&sh->stg_free, (ts - 1) & 1u, sh, 0)) break;
        // 64 columns per round: two loads, one wait; the accumulator is
        // released right after the last round's loads, before its conversion
        bool released = false;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
          const int ma = m0 + c0 + lane, mb = ma + 32;
          const float rs_a = ma < M ? inv_scale[ma] : 0.f, rs_b = mb < M ? inv_scale[mb] : 0.f;
          uint32_t va[32], vb[32];
          tmem_ld32_issue(d_lane + (uint32_t)c0, va);
          tmem_ld32_issue(d_lane + (uint32_t)(c0 + 32), vb);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (c0 + 64 >= c_hi) {
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
              if (h == 0) mbar_arrive(&sh->accum_empty[b]);
              else mbar_arrive_remote(accum_empty_lead);
            }
            released = true;
          }
          // the output type and whether all 64 columns exist are decided once
          // per round, not per value
          auto stage = [&](auto f16, auto full) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float f = __uint_as_float(va[e]) * __shfl_sync(0xffffffffu, rs_a, e);
              const uint16_t o = decltype(f16)::value ? __half_as_ushort(__float2half_rn(f))
                                                      : __bfloat16_as_ushort(__float2bfloat16_rn(f));
              if (decltype(full)::value || c0 + e < c_hi) stg[(c0 + e) * 128 + r] = o;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float f = __uint_as_float(vb[e]) * __shfl_sync(0xffffffffu, rs_b, e);
              const uint16_t o = decltype(f16)::value ? __half_as_ushort(__float2half_rn(f))
                                                      : __bfloat16_as_ushort(__float2bfloat16_rn(f));
              if (decltype(full)::value || c0 + 32 + e < c_hi) stg[(c0 + 32 + e) * 128 + r] = o;
            }
          };
          using T_ = std::true_type;
          using F_ = std::false_type;
          if (c0 + 64 <= c_hi) {
            if (ydt == Q1_F16) stage(T_{}, T_{});
            else stage(F_{}, T_{});
          } else {
            if (ydt == Q1_F16) stage(T_{}, F_{});
            else stage(F_{}, F_{});
          }
        }
        if (!released) {  // no columns for this warp
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            if (h == 0) mbar_arrive(&sh->accum_empty[b]);
            else mbar_arrive_remote(accum_empty_lead);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->stg_ready);
        if (warp == (int)kPairEpiWarp0) {
          int okw = 1;
          if (lane == 0) {
            okw = pair_wait(&sh->stg_ready, ts & 1u, sh, 0);
            if (okw) {
              tma_store_2d(&tmap_y, stg, (t / mtiles) * 256 + 128 * h, m0);
              asm volatile("cp.async.bulk.commit_group;" ::: "memory");
              asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
              mbar_arrive(&sh->stg_free);
            }
          }
          if (!__shfl_sync(0xffffffffu, okw, 0)) break;
        }
        ++ts;
        continue;
      }
      for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(d_lane + (uint32_t)c0, v);
        if (!SPLIT && c0 + 32 >= c_hi) {
          // the accumulator's last columns of this warp are in registers
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            if (h == 0) mbar_arrive(&sh->accum_empty[b]);
            else mbar_arrive_remote(accum_empty_lead);
          }
        }
        if (SPLIT) {
          // partial tile, token-major: column c of this rank's rows
          float *part = reinterpret_cast<float *>(ring);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < NT) part[(size_t)(c0 + e) * 128 + r] = __uint_as_float(v[e]);
        } else {
          const int m_l = m0 + c0 + lane;
          const float rs_l = m_l < M ? inv_scale[m_l] : 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float rs = __shfl_sync(0xffffffffu, rs_l, e);
            const int m = m0 + c0 + e;
            if (c0 + e < c_hi && m < M && n < N) store1(y, (size_t)m * N + n, __uint_as_float(v[e]) * rs, ydt);
          }
        }
      }
      if (!SPLIT && c_lo >= c_hi) {  // no columns for this warp: release at once
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (h == 0) mbar_arrive(&sh->accum_empty[b]);
          else mbar_arrive_remote(accum_empty_lead);
        }
      }
    }
    // the staged tiles' stores complete before the CTA leaves
    if (warp == (int)kPairEpiWarp0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  if (SPLIT) {
    // the pairs' partial tiles are complete in every CTA of the cluster
    cluster_sync_all();
    if (!sh->abort_flag) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int t = t_first;
      const int m0 = (t % mtiles) * NT, nb = (t / mtiles) * 256 + 128 * h;
      const int pr = (int)(crank >> 1);
      // pair pr finishes token columns [NT pr / S, NT (pr + 1) / S) of its half;
      // a thread sums four consecutive weight rows over the S partials in pair order
      const int c_lo = (NT * pr) / ksplit, c_hi = (NT * (pr + 1)) / ksplit;
      const int items = (c_hi - c_lo) * 32;
      for (int i = tid; i < items; i += kPairThreads) {
        const int c = c_lo + (i >> 5), r4 = (i & 31) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p2 = 0; p2 < ksplit; ++p2) {
          const uint32_t src = mapa_rank(smem_u32(ring), (uint32_t)(2 * p2 + h)) + (uint32_t)((c * 128 + r4) * 4);
          float4 v;
          asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                       : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                       : "r"(src)
                       : "memory");
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        const int m = m0 + c, n = nb + r4;
        if (m < M && n < N) {
          const float rs = inv_scale[m];
          const float a4[4] = {acc.x * rs, acc.y * rs, acc.z * rs, acc.w * rs};
          const size_t i0 = (size_t)m * N + n;
          if (n + 4 <= N && (N & 3) == 0) {
            store4(y, i0, a4, ydt);
          } else {
            for (int e = 0; e < 4 && n + e < N; ++e) store1(y, i0 + e, a4[e], ydt);
          }
        }
      }
    }
  }
  cluster_sync_all();  // no CTA releases TMEM or leaves while its pair or cluster still uses it
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// Active clusters of 2 * ksplit pair-kernel CTAs (one CTA per SM).
int pair_clusters(int ksplit) {
  static std::atomic<int> cache[kMaxDevices][5];
  if (ksplit < 1 || ksplit > 4) return 0;
  const int dev = current_device();
  if (dev < kMaxDevices && cache[dev][ksplit].load(std::memory_order_relaxed) > 0)
    return cache[dev][ksplit].load(std::memory_order_relaxed);
  cudaFuncSetAttribute(pair_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmemMax);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * ksplit * 16), 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes(256);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)(2 * ksplit);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, pair_kernel<true, true>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  if (dev < kMaxDevices && n > 0) cache[dev][ksplit].store(n, std::memory_order_relaxed);
  return n;
}

// A launch plan: token tile NT, S pairs per tile (S > 1: cluster split), the
// stream schedule, and the grid (2 CTAs per pair).
struct PairPlan {
  int NT, S;
  bool stream;
  unsigned grid;
};

template <bool SPLIT, bool G128>
cudaError_t launch_pair_g(const WeightView &W, const __half *x16, int64_t M, const float *inv_scale, void *y,
                          const PairPlan &p, float *part, int *cnt, cudaStream_t st, q1_dtype dt) {
  const int NT = p.NT, ksplit = p.S;
  const unsigned grid = p.grid;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)W.K, (cuuint64_t)M};
  cuuint64_t gstride[1] = {(cuuint64_t)W.K * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(NT / 2)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(x16), gdim, gstride, box,
                      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  // 16-bit outputs with 16-byte rows go out through the staging tile and one
  // TMA store per tile (box: 128 weight rows x NT tokens)
  const int ystage = !SPLIT && dt != Q1_F32 && W.N % 8 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0;
  CUtensorMap ymap = map;
  if (ystage) {
    cuuint64_t ydim[2] = {(cuuint64_t)W.N, (cuuint64_t)M};
    cuuint64_t ystr[1] = {(cuuint64_t)W.N * 2};
    cuuint32_t ybox[2] = {128, (cuuint32_t)NT};
    r = encode(&ymap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, y, ydim, ystr, ybox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  static std::atomic<uint64_t> attr{0};
  const int dev = current_device();
  if (not_done(attr, dev)) {
    cudaError_t e = cudaFuncSetAttribute(pair_kernel<SPLIT, G128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPairSmemMax);
    if (e != cudaSuccess) return e;
    mark_done(attr, dev);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kPairThreads, 1, 1);
  cfg.dynamicSmemBytes = pair_smem_bytes(NT);
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = (unsigned)(SPLIT ? 2 * ksplit : 2);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, pair_kernel<SPLIT, G128>, map, ymap, W.w, W.s, W.b, (int)M, (int)W.N, (int)W.K,
                            inv_scale, y, NT, ksplit, W.mbf16 ? 1 : 0, (int)dt, W.gshift, ystage,
                            p.stream ? 1 : 0, part, cnt);
}

// Token-tile width NT (a multiple of 16, at most 256) and the schedule, from
// a cost model in SM clocks fitted to forced plans on GB300: a 128-k step of
// a pair takes about 1024 clocks for any NT up to 256 (8 MMAs of K = 16;
// narrower N does not shorten them, so wide tiles are cheaper per token).
//   round robin (S = 1): whole tiles in rounds over the resident pairs;
//     consecutive single-accumulator tiles are separated by the epilogue
//     stall (~24 NT);
//   cluster split (S = 2..4): S pairs per tile, each a k range, partial
//     tiles summed through distributed shared memory (~48 NT);
//   stream: each pair an equal run of (tile, k-step) units, so the work is
//     spread evenly whatever the tile count; every segment boundary of a run
//     costs ~6 K clocks whatever NT (the accumulator hand-off, or a share's
//     partial-sum write and count), and a shared tile's reduction ~48 NT
//     plus ~24 NT per share read.  The stream plan is taken when the model
//     puts it 0.5 % ahead: forced plans on GB300 agreed with that choice for
//     every shape measured (M from 9 to 4096; 17408 x 5120, 5120 x 17408
//     and 5120 x 5120).
// Ties go to the simpler schedule and the narrower tile.
std::atomic<int> g_plan_nt{0}, g_plan_s{0};

PairPlan plan_pair(int64_t M, int64_t N, int64_t K) {
  const int64_t KS = K / 128, ntn = (N + 255) / 256;
  // the stream schedule indexes (tile, k-step) units with 32-bit integers
  auto stream_fits = [&](int NT) { return ntn * ((M + NT - 1) / NT) * KS < ((int64_t)1 << 31); };
  auto stream_plan = [&](int NT) {
    const int pairs = pair_clusters(1);
    const int64_t T = ntn * ((M + NT - 1) / NT), Wu = T * KS;
    const int64_t P = pairs < Wu ? pairs : Wu;
    return PairPlan{NT, 1, true, (unsigned)(2 * P)};
  };
  {
    const int NT = g_plan_nt.load(std::memory_order_relaxed), S = g_plan_s.load(std::memory_order_relaxed);
    if (NT > 0 && S == 0 && pair_clusters(1) > 0 && stream_fits(NT)) return stream_plan(NT);
    if (NT > 0 && S > 0 && (S == 1 || KS >= 2 * S)) {
      const int clusters = pair_clusters(S);
      if (clusters > 0) {
        const int64_t T = ntn * ((M + NT - 1) / NT);
        return PairPlan{NT, S, false, S > 1 ? (unsigned)(T * 2 * S) : (unsigned)(2 * (T < clusters ? T : clusters))};
      }
    }
  }
  constexpr double kStep = 1024.0;      // clocks per 128-k step of a pair
  constexpr double kEpilogue = 24.0;    // x NT clocks per single-accumulator tile
  constexpr double kReduce = 48.0;      // x NT clocks per split tile (and per share written)
  constexpr double kShareRead = 24.0;   // x NT clocks per share a stream reduction reads
  constexpr double kSegment = 6144.0;   // clocks per segment boundary of a stream run
  PairPlan best{256, 1, false, 0};
  double best_cost = 1e300;
  for (int S = 1; S <= 4; ++S) {
    if (S > 1 && KS < 2 * S) continue;
    const int clusters = pair_clusters(S);
    if (clusters < 1) continue;
    for (int NT = 16; NT <= 256; NT += 16) {
      const int64_t T = ntn * ((M + NT - 1) / NT);
      const int64_t rounds = (T + clusters - 1) / clusters;
      const bool dbuf = S == 1 && NT <= kPairDbufMaxNT;
      const double cost = (double)rounds * ((double)((KS + S - 1) / S) * kStep + (S > 1 ? kReduce * NT : 0.0)) +
                          (dbuf ? 0.0 : (double)(rounds - 1) * kEpilogue * NT);
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = PairPlan{NT, S, false, S > 1 ? (unsigned)(T * 2 * S) : (unsigned)(2 * (T < clusters ? T : clusters))};
      }
    }
  }
  const int pairs = pair_clusters(1);
  if (pairs > 0) {
    for (int NT = 16; NT <= 256; NT += 16) {
      if (!stream_fits(NT)) continue;
      const int64_t T = ntn * ((M + NT - 1) / NT), Wu = T * KS;
      const int64_t P = pairs < Wu ? pairs : Wu;
      const int64_t units = (Wu + P - 1) / P;                  // k-steps of the longest run
      const int64_t segs = (units + KS - 1) / KS + 1;          // segments of a run, at most
      const int64_t shares = (KS + units - 1) / units + 1;     // shares of a tile, at most
      const double cost = (double)units * kStep + (double)(segs - 1) * kSegment + kReduce * NT +
                          kShareRead * NT * (double)shares;
      if (cost < best_cost * 0.995) {
        best_cost = cost;
        best = stream_plan(NT);
      }
    }
  }
  return best;
}

cudaError_t launch_pair(const WeightView &W, const __half *x16, int64_t M, const float *inv_scale, void *y,
                        const PairPlan &p, float *part, int *cnt, cudaStream_t st, q1_dtype dt) {
  if (p.grid == 0) return cudaErrorInvalidConfiguration;
  const bool g128 = W.gshift == 2;
  if (p.S > 1) {
    return g128 ? launch_pair_g<true, true>(W, x16, M, inv_scale, y, p, part, cnt, st, dt)
                : launch_pair_g<true, false>(W, x16, M, inv_scale, y, p, part, cnt, st, dt);
  }
  return g128 ? launch_pair_g<false, true>(W, x16, M, inv_scale, y, p, part, cnt, st, dt)
              : launch_pair_g<false, false>(W, x16, M, inv_scale, y, p, part, cnt, st, dt);
}

// Workspace: fp16 rows [M][K], row scales [M], and for the stream schedule
// the pairs' partial-sum slots (two per pair, NT x 256 fp32 each) and a share
// count per tile half (zeroed by the prep kernel).
struct WideWs {
  size_t x16, scale, part, cnt, total;
};
WideWs wide_ws(int64_t M, int64_t K, const PairPlan &p, int64_t N) {
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  WideWs w{};
  w.x16 = up((size_t)(M * K * 2));
  w.scale = up((size_t)(M * 4));
  if (p.stream) {
    const int64_t T = ((N + 255) / 256) * ((M + p.NT - 1) / p.NT);
    w.part = up((size_t)(p.grid / 2) * 2 * 2 * (size_t)p.NT * 128 * 4);
    w.cnt = up((size_t)T * 2 * 4);
  }
  w.total = w.x16 + w.scale + w.part + w.cnt;
  return w;
}

}  // namespace

void set_pair_plan(int token_tile, int split) {
  const bool ok = token_tile >= 16 && token_tile <= 256 && token_tile % 16 == 0 && split >= 0 && split <= 4;
  g_plan_s.store(ok ? split : 0, std::memory_order_relaxed);
  g_plan_nt.store(ok ? token_tile : 0, std::memory_order_relaxed);
}

size_t wide_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return wide_ws(M, K, plan_pair(M, N, K), N).total;
}

cudaError_t launch_wide(const WeightView &W, const void *x, int64_t M, void *y, void *ws, size_t ws_bytes,
                        cudaStream_t st, q1_dtype dt) {
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  const PairPlan plan = plan_pair(M, W.N, W.K);
  const WideWs w = wide_ws(M, W.K, plan, W.N);
  if (ws_bytes < w.total) return cudaErrorInvalidValue;  // the plan changed since the workspace was sized
  char *wb = static_cast<char *>(ws);
  __half *x16 = reinterpret_cast<__half *>(wb);
  float *inv_scale = reinterpret_cast<float *>(wb + w.x16);
  float *part = plan.stream ? reinterpret_cast<float *>(wb + w.x16 + w.scale) : nullptr;
  int *cnt = plan.stream ? reinterpret_cast<int *>(wb + w.x16 + w.scale + w.part) : nullptr;
  const int ncnt = plan.stream ? (int)(w.cnt / 4) : 0;
  // 1. fp16 rows with per-row power-of-two scales (and the share counts zeroed)
  {
    const unsigned blocks = (unsigned)M;  // one block per row
    const bool held = W.K / 8 <= kPrepHeld * kPrepThreads;
    if (dt == Q1_F32) {
      if (held) x_to_f16_kernel<Q1_F32, true><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
      else x_to_f16_kernel<Q1_F32, false><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
    } else if (dt == Q1_F16) {
      if (held) x_to_f16_kernel<Q1_F16, true><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
      else x_to_f16_kernel<Q1_F16, false><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
    } else {
      if (held) x_to_f16_kernel<Q1_BF16, true><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
      else x_to_f16_kernel<Q1_BF16, false><<<blocks, kPrepThreads, 0, st>>>(x, (int)W.K, x16, inv_scale, cnt, ncnt);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. the pair kernel, launched as a programmatic dependent of the prep:
  //    barrier set-up, TMEM allocation and the first weight stages overlap it
  return launch_pair(W, x16, M, inv_scale, y, plan, part, cnt, st, dt);
}

cudaError_t set_wide_diagnostics(unsigned long long wait_ns, int stall) {
  cudaError_t e = cudaMemcpyToSymbol(c_wide_wait_ns, &wait_ns, sizeof(wait_ns));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(c_wide_stall, &stall, sizeof(stall));
  return e;
}

unsigned int read_and_clear_wide_errors(cudaStream_t st, cudaError_t *err) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_wide_err, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v)
    e = cudaMemcpyToSymbolAsync(g_wide_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (err) *err = e;
  return v;
}

}  // namespace q1
