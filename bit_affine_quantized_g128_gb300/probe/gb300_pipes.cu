// Throughput probes behind the narrow-kernel design (not part of the library):
// mma.sync bf16 / fp8 and binary (AND+popc) MMA rates, LOP3 / IMAD / FFMA
// rates, and back-to-back 12.5 MB streaming launches in a CUDA graph with and
// without programmatic dependent launch.
//
// The MMA loops keep their operands loop-invariant, so they time the MMA
// instructions alone.  For e4m3 that hides the cost that matters: in a real
// kernel whose fp8 operands change every step, ncu's per-opcode counts show
// each m16n8k32 e4m3 mma.sync executing as two HMMAs plus F2FP operand
// conversions on the CUDA cores.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o /tmp/gb300_pipes \
//        bit_affine_quantized_g128_gb300/probe/gb300_pipes.cu && /tmp/gb300_pipes
//
// Every buffer index stays below its allocation (checked on the host before
// the first run: the streaming loop touches at most 16 x 2 x 12533760 bytes of
// a 1 GiB buffer); no kernel waits on anything.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

__global__ void k_mma_bf16(float *out, int iters) {
  float d[4][4] = {};
  uint32_t a0 = threadIdx.x, a1 = a0 * 3, a2 = a0 * 5, a3 = a0 * 7, b0 = a0 ^ 0x3f803f80u, b1 = b0 + 1;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0;
  for (int c = 0; c < 4; ++c)
    for (int j = 0; j < 4; ++j) s += d[c][j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_mma_fp8(float *out, int iters) {
  float d[4][4] = {};
  uint32_t a0 = threadIdx.x * 0x01010101u & 0x3c3c3c3cu, a1 = a0 ^ 0x01010101u, a2 = a0 ^ 0x02020202u,
           a3 = a0 ^ 0x04040404u, b0 = 0x38383838u, b1 = 0x30303030u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0;
  for (int c = 0; c < 4; ++c)
    for (int j = 0; j < 4; ++j) s += d[c][j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_mma_b1(int *out, int iters) {
  int d[4][4] = {};
  uint32_t a0 = threadIdx.x * 0x9E3779B9u, a1 = a0 * 3, b0 = a0 ^ 0x5555u;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k128.row.col.s32.b1.b1.s32.and.popc {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
          : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
          : "r"(a0), "r"(a1), "r"(b0));
  }
  int s = 0;
  for (int c = 0; c < 4; ++c)
    for (int j = 0; j < 4; ++j) s += d[c][j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_lop3(uint32_t *out, int iters) {
  uint32_t v[8];
  for (int j = 0; j < 8; ++j) v[j] = threadIdx.x * (j + 1);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile("lop3.b32 %0, %0, %1, %2, 0xE2;" : "+r"(v[j]) : "r"(0x00010001u << j), "r"(0x3F803F80u));
  }
  uint32_t s = 0;
  for (int j = 0; j < 8; ++j) s ^= v[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_imad(uint32_t *out, int iters) {
  uint32_t v[8];
  for (int j = 0; j < 8; ++j) v[j] = threadIdx.x * (j + 1);
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(v[j]) : "r"(0x01020408u + j), "r"(0x3F80u + j));
  }
  uint32_t s = 0;
  for (int j = 0; j < 8; ++j) s ^= v[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_ffma(float *out, int iters) {
  float v[8];
  for (int j = 0; j < 8; ++j) v[j] = threadIdx.x * (j + 1) * 1e-3f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(v[j]) : "f"(0.999f), "f"(1e-3f));
  }
  float s = 0;
  for (int j = 0; j < 8; ++j) s += v[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// Streams n uint4 words; signals dependents at once and waits for its
// predecessor only at the end (where a decode kernel would read x).
__global__ void k_read_pdl(const uint4 *__restrict__ p, size_t n, uint32_t *out) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    uint4 v = __ldg(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (acc == 0x12345678u) out[0] = acc;
}

int main() {
  int sms = 0, clk_khz = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  const double clk = clk_khz * 1e3;
  int *io;
  uint32_t *uo;
  float *fo;
  cudaMalloc(&io, (size_t)sms * 1024 * 4);
  cudaMalloc(&uo, (size_t)sms * 1024 * 4);
  cudaMalloc(&fo, (size_t)sms * 1024 * 4);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  float ms = 0;
  const int warps = 16, iters = 4096;
  auto rate = [&](double ops) { return ops / sms / (ms * 1e-3 * clk); };
  printf("SMs %d, clock %.0f MHz\n", sms, clk / 1e6);

  k_mma_bf16<<<sms, warps * 32>>>(fo, 16);
  cudaEventRecord(e0);
  k_mma_bf16<<<sms, warps * 32>>>(fo, iters);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("mma.sync m16n8k16 bf16 : %.3f per clk per SM\n", rate((double)sms * warps * iters * 4));

  k_mma_fp8<<<sms, warps * 32>>>(fo, 16);
  cudaEventRecord(e0);
  k_mma_fp8<<<sms, warps * 32>>>(fo, iters);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("mma.sync m16n8k32 e4m3 : %.3f per clk per SM\n", rate((double)sms * warps * iters * 4));

  k_mma_b1<<<sms, warps * 32>>>(io, 16);
  cudaEventRecord(e0);
  k_mma_b1<<<sms, warps * 32>>>(io, iters / 16);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("mma.sync m16n8k128 b1  : %.3f per clk per SM\n", rate((double)sms * warps * (iters / 16) * 4));

  k_lop3<<<sms, 1024>>>(uo, 16);
  cudaEventRecord(e0);
  k_lop3<<<sms, 1024>>>(uo, iters * 4);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("lop3                   : %.1f thread-ops per clk per SM\n", rate((double)sms * 1024 * iters * 4 * 8));

  k_imad<<<sms, 1024>>>(uo, 16);
  cudaEventRecord(e0);
  k_imad<<<sms, 1024>>>(uo, iters * 4);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("imad                   : %.1f thread-ops per clk per SM\n", rate((double)sms * 1024 * iters * 4 * 8));

  k_ffma<<<sms, 1024>>>(fo, 16);
  cudaEventRecord(e0);
  k_ffma<<<sms, 1024>>>(fo, iters * 4);
  cudaEventRecord(e1);
  cudaEventSynchronize(e1);
  cudaEventElapsedTime(&ms, e0, e1);
  printf("ffma                   : %.1f thread-ops per clk per SM\n", rate((double)sms * 1024 * iters * 4 * 8));

  const size_t bytes = (size_t)1 << 30, mat = 12533760, n = mat / 16;
  uint4 *buf;
  cudaMalloc(&buf, bytes);
  cudaMemset(buf, 1, bytes);
  for (int pdl = 0; pdl < 2; ++pdl) {
    cudaStream_t s;
    cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(512);
    cfg.stream = s;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &at;
    cfg.numAttrs = pdl;
    cudaGraph_t g;
    cudaGraphExec_t ge;
    cudaStreamBeginCapture(s, cudaStreamCaptureModeGlobal);
    for (int r = 0; r < 64; ++r)
      cudaLaunchKernelEx(&cfg, k_read_pdl, (const uint4 *)(buf + (size_t)(r % 16) * n * 2), n, uo);
    cudaStreamEndCapture(s, &g);
    cudaGraphInstantiate(&ge, g, 0);
    cudaGraphLaunch(ge, s);
    cudaStreamSynchronize(s);
    cudaEventRecord(e0, s);
    for (int it = 0; it < 10; ++it) cudaGraphLaunch(ge, s);
    cudaEventRecord(e1, s);
    cudaEventSynchronize(e1);
    cudaEventElapsedTime(&ms, e0, e1);
    printf("64 x 12.5 MB reads in a graph, PDL %s: %.2f us per launch, %.1f GB/s\n", pdl ? "on " : "off",
           ms * 1e3 / 640, 640.0 * mat / (ms * 1e-3) / 1e9);
  }
  printf("status: %s\n", cudaGetErrorString(cudaGetLastError()));
  return 0;
}
