// tcgen05 probes for a decode (M <= 8) Q1 kernel with the weights as the A
// operand in tensor memory (not part of the library; the design they describe
// was measured and set aside):
//   1. issue rate of tcgen05.mma.kind::f8f6f4 M=128 N=16 K=32 with A in TMEM,
//      for 1, 2 and 4 issuing warps in one CTA;
//   2. throughput of a one-consumer mbarrier ring (one arrive + one wait per
//      step on each side);
//   3. the pipeline itself: P pipelines per CTA, each four unpack warps (one
//      per TMEM lane quarter, one weight row per thread) and one MMA-issuing
//      warp.  A thread turns each packed word into eight registers of four
//      e4m3 weights (one LOP3 per register against the base 0x38 = 1.0, the
//      selected bit landing in a mantissa or exponent bit), stores them to
//      TMEM with tcgen05.st, and the issuer runs four K=32 MMAs per group of
//      128 k.  Eight groups share one 16-column accumulator through one-hot B
//      columns; the unpack warps read it back every eight groups.  Flags drop
//      parts of the pipeline: 1 = no tcgen05.st, 2 = no MMA, 4 = no waits.
// The packed words come from a shared tile filled once, so no HBM traffic.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o /tmp/tcgen05_decode \
//        bit_affine_quantized_g128_gb300/probe/tcgen05_decode.cu && /tmp/tcgen05_decode
//
// Buffer indices were checked on the host before the first run: TMEM columns
// per CTA are P x (SA x GS x 32 + 32) <= the allocation (static_assert), shared
// tiles are 16 KB + P x 8 KB of a >= 100 KB dynamic allocation, and every
// mbarrier wait is bounded (about 2 s) and aborts the whole CTA on a timeout.
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdint>
#include <vector>
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t *b, unsigned c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(c) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0,1,0,p; }"
               : "=r"(ok) : "r"(smem_u32(b)), "r"(ph) : "memory");
  return ok != 0;
}
__device__ unsigned g_err;
// bounded wait; once any wait of the CTA has timed out every later wait returns false at once
__device__ __forceinline__ bool wait(uint64_t *b, uint32_t ph, volatile int *abort) {
  if (mbar_try(b, ph)) return true;
  if (*abort) return false;
  const long long c0 = clock64();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(b, ph)) return true;
    if ((i & 15u) == 15u && (*abort || clock64() - c0 > 4000000000ll)) { *abort = 1; atomicOr(&g_err, 1u); return false; }
  }
}
template <uint32_t MASK>
__device__ __forceinline__ uint32_t sel(uint32_t src) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(r) : "r"(src), "n"(MASK), "r"(0x38383838u));
  return r;
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
__device__ __forceinline__ void mma_tm(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t acc) {
  constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(16 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p; }"
               ::"r"(d), "r"(a), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void commit(uint64_t *b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
               "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
               ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
               "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
               "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
               "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                 "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
               : "r"(taddr) : "memory");
}

constexpr int kMaxP = 4;
template <int P, int GS, int SA, int COLS, int F = 0>
__global__ void __launch_bounds__(P * 160) pipe(unsigned long long *cyc, float *out, int ngroups) {
  // per pipeline: words tile 128 rows x 16 words (64B swizzle, 8 KB), B tile 8 groups x 2 KB
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);
  uint8_t *btile = base;                 // 16 KB: 8 groups x (16 rows x 128 B)
  uint8_t *wtile = base + 16384;         // P x 8 KB
  __shared__ uint64_t full[kMaxP][SA], empty[kMaxP][SA], dfull[kMaxP][2], dempty[kMaxP][2];
  __shared__ uint32_t tbase;
  __shared__ volatile int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) abort_flag = 0;
  for (int i = tid; i < 16384 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(btile)[i] = (i & 7) == 0 ? 0x30303030u : 0u;
  for (int i = tid; i < P * 8192 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(wtile)[i] = (uint32_t)i * 2654435761u;
  if (tid == 0) {
    for (int p = 0; p < P; ++p) {
      for (int s = 0; s < SA; ++s) { mbar_init(&full[p][s], 4); mbar_init(&empty[p][s], 1); }
      for (int b = 0; b < 2; ++b) { mbar_init(&dfull[p][b], 1); mbar_init(&dempty[p][b], 4); }
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 4 * P) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tbase)), "r"(COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  constexpr uint32_t PCOLS = SA * GS * 32 + 32;  // per pipeline
  const long long t0 = clock64();
  const int nst = ngroups / GS;
  if (warp >= 4 * P) {
    const int p = warp - 4 * P;
    if (lane == 0) {
      const uint32_t A0 = tm + p * PCOLS, D0 = A0 + SA * GS * 32;
      const uint64_t b0 = sw128_desc(smem_u32(btile));
      for (int st = 0; st < nst; ++st) {
        const int s = st % SA;
        if (!(F & 4)) {
          if (!wait(&full[p][s], (uint32_t)(st / SA) & 1u, &abort_flag)) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        }
#pragma unroll
        for (int q = 0; q < GS; ++q) {
          const int g = st * GS + q, blk = g >> 3, gi = g & 7;
          if (!(F & 4) && gi == 0 && blk >= 2) {  // D buffer reuse: epilogue of block blk-2 must be done
            if (!wait(&dempty[p][blk & 1], (uint32_t)((blk >> 1) - 1) & 1u, &abort_flag)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          }
#pragma unroll
          for (int j = 0; j < 4 && !(F & 2); ++j)
            mma_tm(D0 + 16 * (blk & 1), A0 + (s * GS + q) * 32 + 8 * j, b0 + (uint64_t)((gi * 2048 + 32 * j) >> 4),
                   (gi > 0 || j > 0) ? 1u : 0u);
          if (gi == 7) commit(&dfull[p][blk & 1]);
        }
        commit(&empty[p][s]);
        if (abort_flag) break;
      }
      cyc[(blockIdx.x * kMaxP + p) * 2 + 1] = clock64() - t0;
    }
    __syncwarp();
  } else {
    const int p = warp >> 2, wq = warp & 3;
    const int row = 32 * wq + lane;
    const uint32_t A0 = tm + ((uint32_t)(32 * wq) << 16) + p * PCOLS, D0 = A0 + SA * GS * 32;
    const uint8_t *wt = wtile + p * 8192 + row * 64;
    float acc = 0.f;
    for (int st = 0; st < nst; ++st) {
      const int s = st % SA;
      if (!(F & 4) && st >= SA) {
        int ok = 1;
        if (lane == 0) ok = wait(&empty[p][s], (uint32_t)(st / SA - 1) & 1u, &abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      }
#pragma unroll
      for (int q = 0; q < GS; ++q) {
        const int g = st * GS + q;
        const int c = (g & 3) ^ ((row >> 1) & 3);
        const uint4 wv = *reinterpret_cast<const uint4 *>(wt + 16 * c);
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t r[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t x = w4[u], y = w4[u] >> 4;
          r[8 * u + 0] = sel<0x01010101u>(x);
          r[8 * u + 1] = sel<0x02020202u>(x);
          r[8 * u + 2] = sel<0x04040404u>(x);
          r[8 * u + 3] = sel<0x08080808u>(x);
          r[8 * u + 4] = sel<0x01010101u>(y);
          r[8 * u + 5] = sel<0x02020202u>(y);
          r[8 * u + 6] = sel<0x04040404u>(y);
          r[8 * u + 7] = sel<0x08080808u>(y);
        }
        if (!(F & 1)) st32(A0 + (s * GS + q) * 32, r);
        else { uint32_t z = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) z += r[i];
          acc += (float)z; }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[p][s]);
      // epilogue for a finished block of 8 groups (lagging one stage behind)
      const int gend = st * GS + GS;  // groups issued after this stage
      if (!(F & 4) && (gend & 7) == 0 && gend >= 16) {
        const int blk = (gend >> 3) - 2;
        int ok = 1;
        if (lane == 0) ok = wait(&dfull[p][blk & 1], (uint32_t)(blk >> 1) & 1u, &abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        uint32_t v[16];
        ld16(D0 + 16 * (blk & 1), v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int q = 0; q < 8; ++q) acc = fmaf(1.0001f, __uint_as_float(v[2 * q]) + __uint_as_float(v[2 * q + 1]) - 0.5f, acc);
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&dempty[p][blk & 1]);
      }
    }
    out[(blockIdx.x * kMaxP + p) * 128 + row] = acc;
    if (lane == 0 && wq == 0) cyc[(blockIdx.x * kMaxP + p) * 2] = clock64() - t0;
  }
  // all MMAs were committed to barriers that the issuers/epilogue waited on, except the last stages:
  if (warp >= 4 * P && lane == 0) {
    const int p = warp - 4 * P;
    // wait for the last stage's commit (covers every MMA of this issuer)
    if (nst > 0) wait(&empty[p][(nst - 1) % SA], (uint32_t)((nst - 1) / SA) & 1u, &abort_flag);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 4 * P) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(COLS) : "memory");
}


// ---- 1. MMA issue rate with NI issuing warps, each with its own A and D columns
template <int NI>
__global__ void __launch_bounds__(160) mma_issuers(unsigned long long *cyc, int ngroups) {
  __shared__ __align__(1024) uint8_t bt[16 * 128];
  __shared__ uint64_t fin[4];
  __shared__ uint32_t tbase;
  __shared__ volatile int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 16 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(bt)[i] = 0x30303030u;
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < 4; ++i) mbar_init(&fin[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tbase)), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  if (warp < NI && lane == 0) {
    const long long t0 = clock64();
    const uint64_t b0 = sw128_desc(smem_u32(bt));
    const uint32_t A = tm + 32 * warp, D = tm + 256 + 64 * warp;  // cols < 128 and < 512
    for (int g = 0; g < ngroups; ++g) {
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_tm(D + 16 * (g & 3), A + 8 * j, b0 + (uint64_t)((32 * j) >> 4), j > 0);
    }
    commit(&fin[warp]);
    wait(&fin[warp], 0, &abort_flag);
    cyc[blockIdx.x * 4 + warp] = clock64() - t0;
  }
  __syncwarp();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 4) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tm), "r"(512) : "memory");
}

// ---- 2. mbarrier ring: one producer warp, one consumer thread, S slots
template <int S>
__global__ void ring(unsigned long long *cyc, int steps) {
  __shared__ uint64_t full[S], empty[S];
  __shared__ volatile int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const long long t0 = clock64();
  if (warp == 1 && lane == 0) {
    for (int g = 0; g < steps; ++g) {
      if (!wait(&full[g % S], (uint32_t)(g / S) & 1u, &abort_flag)) break;
      mbar_arrive(&empty[g % S]);
    }
    cyc[blockIdx.x] = clock64() - t0;
  } else if (warp == 0) {
    for (int g = 0; g < steps; ++g) {
      int ok = 1;
      if (g >= S && lane == 0) ok = wait(&empty[g % S], (uint32_t)(g / S - 1) & 1u, &abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[g % S]);
    }
  }
}

template <int P, int GS, int SA, int COLS, int F>
void run_pipe(const char *what, int ctas_per_sm, unsigned long long *dc, float *dout) {
  const int ngroups = 8 * 500;
  const int grid = 152 * ctas_per_sm;
  const int dsm = ctas_per_sm == 1 ? 200 * 1024 : 100 * 1024;  // pins the CTAs per SM
  static_assert(P * (SA * GS * 32 + 32) <= COLS, "TMEM columns");
  cudaFuncSetAttribute(pipe<P, GS, SA, COLS, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, dsm);
  pipe<P, GS, SA, COLS, F><<<grid, P * 160, dsm>>>(dc, dout, ngroups);
  pipe<P, GS, SA, COLS, F><<<grid, P * 160, dsm>>>(dc, dout, ngroups);
  const cudaError_t e = cudaDeviceSynchronize();
  unsigned err = 0;
  cudaMemcpyFromSymbol(&err, g_err, 4);
  std::vector<unsigned long long> c(152 * 2 * kMaxP * 2);
  cudaMemcpy(c.data(), dc, c.size() * 8, cudaMemcpyDeviceToHost);
  double worst = 0;
  for (int b = 0; b < grid; ++b)
    for (int p = 0; p < P; ++p)
      for (int r = 0; r < 2; ++r) worst = fmax(worst, (double)c[(b * kMaxP + p) * 2 + r]);
  const double w = (double)ngroups * 16384.0 * P * ctas_per_sm;  // weights per SM
  printf("pipeline %-30s P=%d stage=%d group(s) x %d, %d CTA/SM: %s%s  %.0f clk per group per pipeline, %.1f weights/clk/SM\n",
         what, P, GS, SA, ctas_per_sm, cudaGetErrorString(e), err ? " (wait timed out)" : "", worst / ngroups, w / worst);
}

int main() {
  unsigned long long *dc;
  float *dout;
  cudaMalloc(&dc, 152 * 2 * kMaxP * 2 * 8);
  cudaMalloc(&dout, 152 * 2 * kMaxP * 128 * 4);
  const int NG = 4000;
  {
    auto go = [&](auto kern, int ni) {
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
      kern<<<152, 160, 160 * 1024>>>(dc, NG);
      kern<<<152, 160, 160 * 1024>>>(dc, NG);
      cudaDeviceSynchronize();
      std::vector<unsigned long long> c(152 * 4);
      cudaMemcpy(c.data(), dc, c.size() * 8, cudaMemcpyDeviceToHost);
      double mx = 0;
      for (int i = 0; i < 152; ++i)
        for (int w = 0; w < ni; ++w) mx = fmax(mx, (double)c[i * 4 + w]);
      printf("MMA M128 N16 K32 e4m3, A in TMEM, %d issuing warp(s): %.1f clk per MMA per issuer, %.0f weights/clk/SM\n", ni,
             mx / (4.0 * NG), ni * 4.0 * NG / mx * 4096);
    };
    go(mma_issuers<1>, 1);
    go(mma_issuers<2>, 2);
    go(mma_issuers<4>, 4);
  }
  {
    ring<8><<<152, 64>>>(dc, NG);
    ring<8><<<152, 64>>>(dc, NG);
    cudaDeviceSynchronize();
    unsigned long long c0 = 0;
    cudaMemcpy(&c0, dc, 8, cudaMemcpyDeviceToHost);
    printf("mbarrier ring, 8 slots, one wait + one arrive per step on each side: %.0f clk per step\n", (double)c0 / NG);
  }
  run_pipe<4, 1, 3, 512, 0>("full", 1, dc, dout);
  run_pipe<4, 1, 3, 512, 4>("no waits", 1, dc, dout);
  run_pipe<4, 1, 3, 512, 3>("waits only (no st, no MMA)", 1, dc, dout);
  run_pipe<4, 1, 3, 512, 6>("st only (no MMA, no waits)", 1, dc, dout);
  run_pipe<2, 2, 3, 512, 0>("full", 1, dc, dout);
  run_pipe<2, 1, 3, 256, 0>("full", 2, dc, dout);
  run_pipe<1, 2, 3, 256, 0>("full", 1, dc, dout);
  return 0;
}
