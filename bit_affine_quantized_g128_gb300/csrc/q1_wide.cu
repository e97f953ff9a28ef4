// Wide (prefill) Q1 matmul on the tcgen05 tensor cores:
//   y[M][N] = x[M][K] . Wd^T, fp32 accumulation in tensor memory.
//
// The page "Support Bonsai-27B affine Q1" (higgs PR #212), section
// "Limitations / non-goals", runs forwards wider than the narrow threshold by
// dequantizing the whole matrix to the input dtype and calling a dense matmul,
// which is what set its peak memory ("Measured impact": peak about 6.65 GB
// from dense prefill temporaries).  Here the dequantization happens per tile
// in shared memory, feeding the MMA directly: no dense weight temporary.
//
// Operand precision.  Rounding the dequantized weights to bf16 (a half-ulp of
// 2^-8, the same for every weight of a symmetric group) moves a few outputs in
// 10^5 past the per-element error bar the method is held to, so the tiles are
// fp16 instead: symmetric weights +-s/2 are exact in fp16 and affine values
// s+b are rounded once at 2^-11.  The activations go to fp16 through a
// per-row power-of-two scale 2^e_m chosen so that the row maximum lands in
// [2^14, 2^15) (exact for every normal fp16 result, no overflow); the
// epilogue multiplies by 2^-e_m.  A small prep kernel writes the scaled fp16
// rows and the scales into the caller's workspace.
//
// One CTA computes MT x 128 tokens x 256 rows (MT = 2 when that needs fewer
// CTA-times than MT = 1, see launch_wide):
// every dequantized weight tile feeds MT MMAs, one per 128-token tile, into
// MT 256-column TMEM accumulators.  About 192 KB of shared memory keeps the
// CTA alone on its SM, so its TMEM allocation (256 or 512 columns) cannot
// contend:
//   warp 0        TMA producer: x tiles [MT x 128 tokens x 64 k] fp16, 128B swizzle
//   warp 1        TMEM allocator and the single MMA-issuing thread
//                 (tcgen05.mma.cta_group::1.kind::f16, M=128 N=256 K=16)
//   warps 2..17   dequantizers: two threads per weight row read the packed
//                 words of one group (uint4) and the group's scale/bias; each
//                 writes 32 fp16 (one word) per k-step into the 128B-swizzled
//                 K-major layout the MMA reads; then the epilogue:
//                 TMEM -> registers -> scale -> bf16 -> global.
// Stages: 4 (MT = 1) or 3 (MT = 2) x (x tiles + 32 KB weight tile), mbarrier
// hand-offs.
// When the tiles are too few to fill the SMs (small M, or the 5120-row down
// projection), a cluster of up to 8 CTAs splits K for each tile and sums the
// partial tiles through distributed shared memory (see SPLIT below).
// Every wait is bounded (globaltimer); one that runs out sets a device error
// word and a CTA-wide abort flag so that the other roles stop waiting too.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace q1 {

__device__ unsigned int g_wide_err = 0;

namespace {

constexpr int BM = 128;  // tokens per MMA tile (TMEM lanes)
constexpr int BN = 256;  // weight rows per tile (MMA N)
constexpr int BK = 64;   // k per stage (one 128-byte swizzle atom of fp16)
// MT token tiles of BM per CTA share every dequantized weight tile (MT = 2
// halves the dequantization per MMA); the stages then shrink from 4 to 3
template <int MT> constexpr int kStages = MT == 1 ? 4 : 3;
constexpr int kThreadsWide = 576;  // 18 warps
constexpr int kDeqWarp0 = 2;
constexpr int kDeqThreads = 512;   // two threads per weight row: one word each per k-step
constexpr uint32_t A_TILE = BM * BK * 2;   // 16 KB per token tile
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

constexpr int kMaxStages = 4;
// split-K partial tile in the (then idle) stage memory: 128 rows x 256 fp32,
// rows padded by 16 bytes so that a warp's row-wise stores spread over the banks
constexpr int kPartStride = BN + 4;
struct __align__(8) WideShared {
  uint64_t full_a[kMaxStages];
  uint64_t full_b[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t accum_full;
  uint32_t tmem_base;
  volatile int abort_flag;
};

template <int MT>
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages<MT> * (MT * A_TILE + B_BYTES) + sizeof(WideShared);

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

// Bounded wait on the phase with the given parity.  Returns false when the
// wait ran out or another role of this CTA already aborted.
__device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, WideShared *sh) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try(addr, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(addr, parity)) return true;
    if ((i & 15u) == 15u) {
      if (sh->abort_flag) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        sh->abort_flag = 1;
        atomicOr(&g_wide_err, 1u);
        return false;
      }
    }
  }
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

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4..5 = 1), fp16 A
// and B (format 0 at bits 7..9 and 10..12), both K-major, N >> 3 at bits
// 17..22, M >> 4 at bits 24..28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 32 weights of one word -> 16 bf16x2 in k order: out[j] = (k = 2j, 2j+1).
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
// eight values, y + i aligned to 16 bytes
__device__ __forceinline__ void store8(void *y, size_t i, const float (&f)[8], int dt) {
  if (dt == Q1_F32) {
    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(y) + i);
    d[0] = make_float4(f[0], f[1], f[2], f[3]);
    d[1] = make_float4(f[4], f[5], f[6], f[7]);
  } else {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(y) + i) =
        make_uint4(pack2(f[0], f[1], dt), pack2(f[2], f[3], dt), pack2(f[4], f[5], dt), pack2(f[6], f[7], dt));
  }
}

// One thread's share of a 128-k unit: its row's four words, and the metadata
// of the two words it expands (k-steps 0 and 1); the same group for both
// unless the group size is 32 or 64.
struct GroupData {
  uint4 w;
  uint16_t s[2], b[2];
};

// SPLIT: a thread-block cluster of `ksplit` CTAs shares one output tile, each
// taking a contiguous range of the 128-k groups; the fp32 partial tiles are
// summed through distributed shared memory in rank order (deterministic, no
// workspace).  Only with MT = 1.
template <int MT, bool SPLIT, bool G128>
__global__ void __launch_bounds__(kThreadsWide, 1)
wide_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint32_t *__restrict__ W,
            const uint16_t *__restrict__ S, const uint16_t *__restrict__ Bv, int M, int N, int K,
            const float *__restrict__ inv_scale, void *__restrict__ y, int ksplit, int mbf16, int ydt,
            int gshift) {
  static_assert(!SPLIT || MT == 1, "split-K keeps one token tile per CTA");
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int STAGES = kStages<MT>;
  constexpr uint32_t A_BYTES = MT * A_TILE;        // the stage's x tiles (MT x 128 tokens)
  constexpr uint32_t kTmemCols = 256 * MT;         // one 256-column accumulator per token tile
  unsigned char *sa = base;                        // STAGES x A_BYTES
  unsigned char *sb = base + STAGES * A_BYTES;     // STAGES x B_BYTES
  WideShared *sh = reinterpret_cast<WideShared *>(sb + STAGES * B_BYTES);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = SPLIT ? (int)(blockIdx.x % (unsigned)ksplit) : 0;
  const int n0 = (SPLIT ? (int)(blockIdx.x / (unsigned)ksplit) : (int)blockIdx.x) * BN;
  const int m0 = blockIdx.y * (BM * MT);
  // this CTA's groups [g_lo, g_hi) and k-steps (two per group)
  const int GK = K / 128;
  const int g_lo = SPLIT ? (int)(((int64_t)GK * rank) / ksplit) : 0;
  const int g_hi = SPLIT ? (int)(((int64_t)GK * (rank + 1)) / ksplit) : GK;
  const int KS0 = 2 * g_lo, KSTEPS = 2 * (g_hi - g_lo);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full_a[s], 1);
      mbar_init(&sh->full_b[s], kDeqThreads / 32);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->accum_full, 1);
    sh->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem_d = sh->tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer (x tiles)
    if (lane == 0) {
      // the fp16 rows come from the prep kernel that precedes this one
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int s = ks % STAGES;
        const uint32_t ph = (uint32_t)(ks / STAGES) & 1u;
        if (!mbar_wait(&sh->empty[s], ph ^ 1u, sh)) break;
        mbar_arrive_expect_tx(&sh->full_a[s], A_BYTES);
        tma_load_2d(sa + s * A_BYTES, &tmap_x, &sh->full_a[s], (KS0 + ks) * BK, m0);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int ks = 0; ks < KSTEPS && ok; ++ks) {
        const int s = ks % STAGES;
        const uint32_t ph = (uint32_t)(ks / STAGES) & 1u;
        ok = mbar_wait(&sh->full_a[s], ph, sh) && mbar_wait(&sh->full_b[s], ph, sh);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = smem_u32(sa + s * A_BYTES), b_addr = smem_u32(sb + s * B_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            umma_bf16(tmem_d + 256u * mt, sw128_desc(a_addr + mt * A_TILE + kk * 32), sw128_desc(b_addr + kk * 32),
                      (ks > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&sh->empty[s]);
      }
      umma_commit(&sh->accum_full);  // arrives once every issued MMA has completed
    }
  } else {
    // ---------------- dequantizers: threads 2r and 2r+1 own weight row n0 + r;
    //                  thread 2r+wh expands word wh of each 64-k stage
    const int d = (tid - kDeqWarp0 * 32) >> 1, wh = tid & 1;
    const int n = n0 + d;
    const bool ok_row = n < N;
    const int wpr = K / 32, G = wpr >> gshift;  // G: metadata groups per row
    const uint4 *wrow = reinterpret_cast<const uint4 *>(W + (size_t)(ok_row ? n : 0) * wpr);
    const uint16_t *srow = S + (size_t)(ok_row ? n : 0) * G;
    const uint16_t *brow = Bv ? Bv + (size_t)(ok_row ? n : 0) * G : nullptr;
    auto load = [&](int g, GroupData &gd) {  // g: 128-k unit
      if (g < g_hi && ok_row) {
        gd.w = __ldg(wrow + g);
        if constexpr (G128) {  // one group per 128-k unit
          gd.s[0] = gd.s[1] = srow[g];
          gd.b[0] = gd.b[1] = brow ? brow[g] : (uint16_t)0;
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int mi = (4 * g + 2 * h + wh) >> gshift;  // group of word 2h + wh
            gd.s[h] = srow[mi];
            gd.b[h] = brow ? brow[mi] : (uint16_t)0;
          }
        }
      } else {
        gd.w = make_uint4(0, 0, 0, 0);
        gd.s[0] = gd.s[1] = gd.b[0] = gd.b[1] = 0;
      }
    };
    bool alive = true;
    // fp16x2 patterns of the two dequantized values (q = 0, q = 1) of a group
    auto pair_of = [&](uint16_t s16, uint16_t b16, uint32_t &lo2, uint32_t &hi2) {
      const float sc = meta_f32(s16, mbf16 != 0);
      const float bi = brow ? meta_f32(b16, mbf16 != 0) : __fmul_rn(-0.5f, sc);
      const uint32_t lo16 = __half_as_ushort(__float2half_rn(bi));
      const uint32_t hi16 = __half_as_ushort(__float2half_rn(__fadd_rn(sc, bi)));
      lo2 = lo16 | (lo16 << 16);
      hi2 = hi16 | (hi16 << 16);
    };
    auto process = [&](int g, const GroupData &gd) {
      uint32_t lo2v[2], hi2v[2];
      pair_of(gd.s[0], gd.b[0], lo2v[0], hi2v[0]);
      if constexpr (G128) {
        lo2v[1] = lo2v[0];
        hi2v[1] = hi2v[0];
      } else {
        pair_of(gd.s[1], gd.b[1], lo2v[1], hi2v[1]);
      }
      if constexpr (MT == 2) {
        // the group's two k-steps, one stage at a time: each stage is handed to
        // the MMA as soon as it is written, so that the dequantizers can run up
        // to STAGES stages ahead
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ks = 2 * (g - g_lo) + h;  // this CTA's k-step
          const int st = ks % STAGES;
          const uint32_t ph = (uint32_t)(ks / STAGES) & 1u;
          // one lane waits, the warp follows its verdict (keeps the warp converged)
          int okw = 0;
          if (lane == 0) okw = alive && mbar_wait(&sh->empty[st], ph ^ 1u, sh);
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) {
            alive = false;
            return;
          }
          unsigned char *rowp = sb + st * B_BYTES + d * 128;
          const uint32_t word = h == 0 ? (wh == 0 ? gd.w.x : gd.w.y) : (wh == 0 ? gd.w.z : gd.w.w);
          uint32_t out[16];
          expand_word(word, lo2v[h], hi2v[h], out);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = wh * 4 + q;  // 16-byte chunk: k = 8c .. 8c+7 of this stage
            *reinterpret_cast<uint4 *>(rowp + ((c ^ (d & 7)) << 4)) =
                make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh->full_b[st]);
        }
      } else {
        // four stages: wait for both of the group's stages, write both, then
        // one proxy fence and the two arrivals (halves the hand-offs; with four
        // stages the dequantizers still run a stage ahead)
        const int ks0 = 2 * (g - g_lo);  // this CTA's k-step
        const int s0 = ks0 % STAGES, s1 = (ks0 + 1) % STAGES;
        const uint32_t ph0 = (uint32_t)(ks0 / STAGES) & 1u, ph1 = (uint32_t)((ks0 + 1) / STAGES) & 1u;
        // one lane waits, the warp follows its verdict (keeps the warp converged)
        int okw = 0;
        if (lane == 0)
          okw = alive && mbar_wait(&sh->empty[s0], ph0 ^ 1u, sh) && mbar_wait(&sh->empty[s1], ph1 ^ 1u, sh);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          alive = false;
          return;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          unsigned char *rowp = sb + (h == 0 ? s0 : s1) * B_BYTES + d * 128;
          const uint32_t word = h == 0 ? (wh == 0 ? gd.w.x : gd.w.y) : (wh == 0 ? gd.w.z : gd.w.w);
          uint32_t out[16];
          expand_word(word, lo2v[h], hi2v[h], out);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = wh * 4 + q;  // 16-byte chunk: k = 8c .. 8c+7 of this stage
            *reinterpret_cast<uint4 *>(rowp + ((c ^ (d & 7)) << 4)) =
                make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh->full_b[s0]);
          mbar_arrive(&sh->full_b[s1]);
        }
      }
    };
    GroupData r0, r1, r2;
    load(g_lo, r0);
    load(g_lo + 1, r1);
    for (int g = g_lo; g < g_hi && alive; g += 3) {
      load(g + 2, r2);
      process(g, r0);
      if (g + 1 >= g_hi || !alive) break;
      load(g + 3, r0);
      process(g + 1, r1);
      if (g + 2 >= g_hi || !alive) break;
      load(g + 4, r1);
      process(g + 2, r2);
    }

    // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4).., columns half (w-2)/4
    int acc_ok = 0;
    if (lane == 0) acc_ok = mbar_wait(&sh->accum_full, 0u, sh) && !sh->abort_flag;
    acc_ok = __shfl_sync(0xffffffffu, acc_ok, 0);
    if (acc_ok) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      asm volatile("griddepcontrol.wait;" ::: "memory");  // inv_scale comes from the prep kernel
      const int quarter = warp & 3, part = (warp - kDeqWarp0) >> 2;  // 4 column quarters
#pragma unroll 1
      for (int mc = 0; mc < 2 * MT; ++mc) {
        const int mt = mc >> 1, cc = mc & 1;
        const int m = m0 + BM * mt + 32 * quarter + lane;
        const float rs = m < M ? inv_scale[m] : 0.f;
        const int col = part * 64 + cc * 32;
        uint32_t v[32];
        const uint32_t taddr = tmem_d + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(256 * mt + col);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
              "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
              "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
              "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
              "=r"(v[31])
            : "r"(taddr)
            : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (SPLIT) {
          // this rank's partial sums stay in shared memory for the cluster reduction
          float *prow = reinterpret_cast<float *>(sa) + (size_t)(32 * quarter + lane) * kPartStride + col;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(prow + 4 * q) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        } else if (m < M) {
          const int n = n0 + col;
          const size_t i0 = (size_t)m * N + n;
          // 16-byte stores need 16-byte aligned rows: N % 8 == 0 (16-bit
          // outputs) or N % 4 == 0 (fp32)
          if (n + 32 <= N && (N & (ydt == Q1_F32 ? 3 : 7)) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(v[8 * q + e]) * rs;
              store8(y, i0 + 8 * q, f, ydt);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (n + e < N) store1(y, i0 + e, __uint_as_float(v[e]) * rs, ydt);
          }
        }
      }
    }
  }

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (SPLIT) {
    // rank r finishes rows [128 r / S, 128 (r+1) / S) of the tile: the sum of
    // the ranks' partial tiles in rank order, scaled back and rounded once
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    cluster.sync();
    asm volatile("griddepcontrol.wait;" ::: "memory");  // inv_scale comes from the prep kernel
    const int r_lo = (BM * rank) / ksplit, r_hi = (BM * (rank + 1)) / ksplit;
    const int nvec = (r_hi - r_lo) * (BN / 4);
    for (int i = tid; i < nvec; i += kThreadsWide) {
      const int r = r_lo + i / (BN / 4), c4 = i % (BN / 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q = 0; q < ksplit; ++q) {
        const float *pq = cluster.map_shared_rank(reinterpret_cast<float *>(sa), q);
        const float4 v = *reinterpret_cast<const float4 *>(pq + (size_t)r * kPartStride + 4 * c4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const int m = m0 + r, n = n0 + 4 * c4;
      if (m < M && n < N) {
        const float rs = inv_scale[m];
        const size_t i0 = (size_t)m * N + n;
        const float a4[4] = {acc.x * rs, acc.y * rs, acc.z * rs, acc.w * rs};
        if (n + 4 <= N && (N & 3) == 0) {
          store4(y, i0, a4, ydt);
        } else {
          for (int e = 0; e < 4 && n + e < N; ++e) store1(y, i0 + e, a4[e], ydt);
        }
      }
    }
    cluster.sync();  // no rank leaves while another still reads its partial tile
  }
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d), "r"(kTmemCols)
                 : "memory");
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
// number, and rounds fp32 activations once (2^-11).  One warp per row.
template <int XDT>
__global__ void __launch_bounds__(256) x_to_f16_kernel(const void *__restrict__ x, int M,
                                                       int K, __half *__restrict__ x16,
                                                       float *__restrict__ inv_scale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M) return;
  const void *row = static_cast<const char *>(x) + (size_t)warp * K * (XDT == Q1_F32 ? 4 : 2);
  const int n8 = K / 8;  // chunks of 8 activations
  float mx = 0.f;
  for (int i = lane; i < n8; i += 32) {
    float f[8];
    load8<XDT>(row, i, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  int e = 0;
  if (mx > 0.f && mx <= 3.0e38f) {
    const int E = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2) for normal mx
    e = 14 - (E < -126 ? -126 : E);
    if (e > 126) e = 126;
    if (e < -126) e = -126;
  }
  const float sc = __uint_as_float((uint32_t)(127 + e) << 23);   // 2^e, exact
  const float isc = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, exact
  uint4 *out = reinterpret_cast<uint4 *>(x16 + (size_t)warp * K);
  for (int i = lane; i < n8; i += 32) {
    float f[8];
    load8<XDT>(row, i, f);
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(f[2 * q] * sc, f[2 * q + 1] * sc);
      o[q] = *reinterpret_cast<const uint32_t *>(&h);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) inv_scale[warp] = isc;
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

template <int MT, bool SPLIT, bool G128>
cudaError_t launch_wide_mma_g(const WeightView &W, const __half *x16, int64_t M, const float *inv_scale, void *y,
                            int ksplit, cudaStream_t st, q1_dtype dt) {
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)W.K, (cuuint64_t)M};
  cuuint64_t gstride[1] = {(cuuint64_t)W.K * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)(BM * MT)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(x16), gdim, gstride, box,
                      estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> attr{0};
  const int dev = current_device();
  if (not_done(attr, dev)) {
    cudaError_t e = cudaFuncSetAttribute(wide_kernel<MT, SPLIT, G128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes<MT>);
    if (e != cudaSuccess) return e;
    mark_done(attr, dev);
  }
  const unsigned ntn = (unsigned)((W.N + BN - 1) / BN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntn * (unsigned)(SPLIT ? ksplit : 1), (unsigned)((M + BM * MT - 1) / (BM * MT)), 1);
  cfg.blockDim = dim3(kThreadsWide, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes<MT>;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = (unsigned)(SPLIT ? ksplit : 1);
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = SPLIT ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, wide_kernel<MT, SPLIT, G128>, map, W.w, W.s, W.b, (int)M, (int)W.N, (int)W.K,
                            inv_scale, y, SPLIT ? ksplit : 1, W.mbf16 ? 1 : 0, (int)dt, W.gshift);
}

// 128-groups (one scale per 128-k unit) compile to their own kernel: the
// per-word metadata of 32- and 64-groups costs the dequantizers ~5 %.
template <int MT, bool SPLIT>
cudaError_t launch_wide_mma(const WeightView &W, const __half *x16, int64_t M, const float *inv_scale, void *y,
                            int ksplit, cudaStream_t st, q1_dtype dt) {
  if (W.gshift == 2) return launch_wide_mma_g<MT, SPLIT, true>(W, x16, M, inv_scale, y, ksplit, st, dt);
  return launch_wide_mma_g<MT, SPLIT, false>(W, x16, M, inv_scale, y, ksplit, st, dt);
}

// Clusters of `ks` split-K CTAs that can be resident at once (one per SM).
int wide_split_clusters(int ks) {
  static std::atomic<int> cache[kMaxDevices][9];
  if (ks < 2 || ks > 8) return 0;
  const int dev = current_device();
  if (dev < kMaxDevices && cache[dev][ks].load(std::memory_order_relaxed) > 0)
    return cache[dev][ks].load(std::memory_order_relaxed);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ks * 32), 1, 1);
  cfg.blockDim = dim3(kThreadsWide, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes<1>;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)ks;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaFuncSetAttribute(wide_kernel<1, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes<1>);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, wide_kernel<1, true, true>, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 0;
  }
  if (dev < kMaxDevices && n > 0) cache[dev][ks].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

size_t wide_workspace_bytes(int64_t M, int64_t K) {
  const size_t x16 = ((size_t)(M * K * 2) + 255) / 256 * 256;
  return x16 + ((size_t)(M * 4) + 255) / 256 * 256;
}

cudaError_t launch_wide(const WeightView &W, const void *x, int64_t M, void *y, void *ws,
                        cudaStream_t st, q1_dtype dt) {
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  __half *x16 = static_cast<__half *>(ws);
  float *inv_scale = reinterpret_cast<float *>(static_cast<char *>(ws) +
                                               ((size_t)(M * W.K * 2) + 255) / 256 * 256);
  // 1. fp16 rows with per-row power-of-two scales
  {
    const unsigned blocks = (unsigned)((M * 32 + 255) / 256);
    if (dt == Q1_F32) x_to_f16_kernel<Q1_F32><<<blocks, 256, 0, st>>>(x, (int)M, (int)W.K, x16, inv_scale);
    else if (dt == Q1_F16) x_to_f16_kernel<Q1_F16><<<blocks, 256, 0, st>>>(x, (int)M, (int)W.K, x16, inv_scale);
    else x_to_f16_kernel<Q1_BF16><<<blocks, 256, 0, st>>>(x, (int)M, (int)W.K, x16, inv_scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // 2. the tcgen05 kernel, launched as a programmatic dependent of the prep:
  //    barrier set-up, TMEM allocation and the first weight tiles overlap it.
  //    Two token tiles per CTA when that takes fewer CTA-times: one CTA runs
  //    per SM, a CTA with two tiles takes ~1.5x the time of one with a single
  //    tile (measured), and the waves are whole.
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int64_t ntiles = (W.N + BN - 1) / BN;
  const int64_t tiles1 = ntiles * ((M + BM - 1) / BM);
  // Cost in CTA-times of a single-tile CTA over all of K: whole waves of
  // resident CTAs (one per SM) x the time of one CTA.  A CTA with two token
  // tiles takes ~1.5x (measured); a split-K CTA 1/S of it plus its share of
  // the cluster reduction.
  double best = (double)((tiles1 + sms - 1) / sms);
  int mode = 1, best_split = 1;
  if (M > BM) {
    const int64_t tiles2 = ntiles * ((M + 2 * BM - 1) / (2 * BM));
    const double c2 = 1.5 * (double)((tiles2 + sms - 1) / sms);
    if (c2 < best) {
      best = c2;
      mode = 2;
    }
  }
  const int GK = (int)(W.K / 128);
  for (int ks = 2; ks <= 8 && ks <= GK / 2; ++ks) {
    const int active = wide_split_clusters(ks);
    if (active < 1) continue;
    const double c = (double)((tiles1 + active - 1) / active) * (1.0 / ks + 0.05);
    if (c < 0.9 * best) {
      best = c;
      mode = 3;
      best_split = ks;
    }
  }
  if (mode == 2) return launch_wide_mma<2, false>(W, x16, M, inv_scale, y, 1, st, dt);
  if (mode == 3) return launch_wide_mma<1, true>(W, x16, M, inv_scale, y, best_split, st, dt);
  return launch_wide_mma<1, false>(W, x16, M, inv_scale, y, 1, st, dt);
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
