// Elementwise Q1 kernels: pack, unpack, dequantize, embedding gather and the
// symmetric-metadata check.  All of them are HBM-bound streams: one thread per
// packed 32-bit word, 16-byte loads/stores, grid-stride loops over a grid
// sized in multiples of the SM count.
//
// Definitions: "1-bit affine weight support" (rMLX issue #207), "The good news -
// packing is standard" (32 weights per uint32, fp16 scales/biases per group of
// 128, bit 0 -> negative, bit 1 -> positive); "Support Bonsai-27B affine Q1"
// (higgs PR #212), "What" (w = scale*q + bias, symmetric bias = -scale/2) and
// the walkthrough's "symmetric bias compaction and validation".
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q1_internal.h"

namespace q1 {
namespace {

int sm_count() {
  static int cached = 0;
  if (cached == 0) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached = n > 0 ? n : 148;
  }
  return cached;
}

unsigned grid_for(int64_t items, int threads) {
  int64_t want = (items + threads - 1) / threads;
  int64_t cap = (int64_t)sm_count() * 16;  // 16 resident 256-thread blocks' worth per SM
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (unsigned)want;
}

// Four 0/1 bytes (bit 0 of each byte) -> a 4-bit nibble, byte j -> bit j.
// The multiplier moves bit 8j to bit 24+j; every other partial product lands
// outside bits 24..27 and no two land on the same bit, so nothing carries in.
__device__ __forceinline__ uint32_t bytes_to_nibble(uint32_t v) {
  return (((v & 0x01010101u) * 0x01020408u) >> 24) & 0xFu;
}

// A 4-bit nibble -> four 0/1 bytes, bit j -> byte j.  The multiplier puts bit
// j at positions j, j+7, j+14, j+21 (all distinct, no carries); bit j lands on
// 8j exactly when the shift is 7j.
__device__ __forceinline__ uint32_t nibble_to_bytes(uint32_t v) {
  return ((v & 0xFu) * 0x00204081u) & 0x01010101u;
}

__global__ void pack_kernel(const uint8_t *__restrict__ bits, uint32_t *__restrict__ w,
                            int64_t nwords) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 *src = reinterpret_cast<const uint4 *>(bits + i * 32);
    uint4 a = src[0], b = src[1];
    uint32_t r = bytes_to_nibble(a.x) | (bytes_to_nibble(a.y) << 4) |
                 (bytes_to_nibble(a.z) << 8) | (bytes_to_nibble(a.w) << 12) |
                 (bytes_to_nibble(b.x) << 16) | (bytes_to_nibble(b.y) << 20) |
                 (bytes_to_nibble(b.z) << 24) | (bytes_to_nibble(b.w) << 28);
    w[i] = r;
  }
}

__global__ void unpack_kernel(const uint32_t *__restrict__ w, uint8_t *__restrict__ bits,
                              int64_t nwords) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t v = w[i];
    uint4 a, b;
    a.x = nibble_to_bytes(v);
    a.y = nibble_to_bytes(v >> 4);
    a.z = nibble_to_bytes(v >> 8);
    a.w = nibble_to_bytes(v >> 12);
    b.x = nibble_to_bytes(v >> 16);
    b.y = nibble_to_bytes(v >> 20);
    b.z = nibble_to_bytes(v >> 24);
    b.w = nibble_to_bytes(v >> 28);
    uint4 *dst = reinterpret_cast<uint4 *>(bits + i * 32);
    dst[0] = a;
    dst[1] = b;
  }
}

// fp32 dequantized pair for one (row, group): lo = bias (q = 0),
// hi = fl32(scale + bias) (q = 1).  Symmetric: bias = -scale/2 in fp32 (exact).
__device__ __forceinline__ void group_values(const uint16_t *__restrict__ s,
                                             const uint16_t *__restrict__ b, int64_t idx,
                                             float &lo, float &hi) {
  float sc = __half2float(__ushort_as_half(s[idx]));
  float bi = b ? __half2float(__ushort_as_half(b[idx])) : __fmul_rn(-0.5f, sc);
  lo = bi;
  hi = __fadd_rn(sc, bi);
}

// 32 outputs of one word, as 16-bit patterns lo16 / hi16 selected by the bits.
__device__ __forceinline__ void store_word_16(uint16_t lo16, uint16_t hi16, uint32_t word,
                                              uint4 *dst) {
  uint32_t out[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    uint32_t a = (word >> (2 * j)) & 1u ? hi16 : lo16;
    uint32_t c = (word >> (2 * j + 1)) & 1u ? hi16 : lo16;
    out[j] = a | (c << 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[j] = make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
}

__device__ __forceinline__ void store_word_f32(float lo, float hi, uint32_t word, uint4 *dst) {
  uint32_t lo32 = __float_as_uint(lo), hi32 = __float_as_uint(hi);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 v;
    v.x = (word >> (4 * j + 0)) & 1u ? hi32 : lo32;
    v.y = (word >> (4 * j + 1)) & 1u ? hi32 : lo32;
    v.z = (word >> (4 * j + 2)) & 1u ? hi32 : lo32;
    v.w = (word >> (4 * j + 3)) & 1u ? hi32 : lo32;
    dst[j] = v;
  }
}

template <int OUT>  // 0 = bf16, 1 = f16, 2 = f32
__device__ __forceinline__ void emit_word(float lo, float hi, uint32_t word, void *out_row,
                                          int64_t c) {
  if (OUT == 2) {
    store_word_f32(lo, hi, word, reinterpret_cast<uint4 *>(static_cast<float *>(out_row) + c * 32));
  } else {
    uint16_t l16, h16;
    if (OUT == 0) {
      l16 = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
      h16 = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    } else {
      l16 = __half_as_ushort(__float2half_rn(lo));
      h16 = __half_as_ushort(__float2half_rn(hi));
    }
    store_word_16(l16, h16, word,
                  reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out_row) + c * 32));
  }
}

template <int OUT>
__global__ void dequantize_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                                  const uint16_t *__restrict__ b, int64_t N, int64_t K,
                                  void *__restrict__ out) {
  const int64_t wpr = K / 32, G = K / 128, nwords = N * wpr;
  const int esz = OUT == 2 ? 4 : 2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t n = i / wpr, c = i - n * wpr;
    float lo, hi;
    group_values(s, b, n * G + c / 4, lo, hi);
    emit_word<OUT>(lo, hi, w[i], static_cast<char *>(out) + n * K * esz, c);
  }
}

template <int OUT>
__global__ void gather_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                              const uint16_t *__restrict__ b, int64_t V, int64_t K,
                              const int32_t *__restrict__ ids, int64_t T, void *__restrict__ out,
                              int32_t *__restrict__ bad) {
  const int64_t wpr = K / 32, G = K / 128, nwords = T * wpr;
  const int esz = OUT == 2 ? 4 : 2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nwords;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = i / wpr, c = i - t * wpr;
    int64_t row = ids[t];
    char *out_row = static_cast<char *>(out) + t * K * esz;
    if (row < 0 || row >= V) {
      uint4 *dst = reinterpret_cast<uint4 *>(out_row + c * 32 * esz);
      const int n16 = 32 * esz / 16;
      for (int j = 0; j < n16; ++j) dst[j] = make_uint4(0, 0, 0, 0);
      if (c == 0 && bad) atomicAdd(bad, 1);
      continue;
    }
    float lo, hi;
    group_values(s, b, row * G + c / 4, lo, hi);
    emit_word<OUT>(lo, hi, w[row * wpr + c], out_row, c);
  }
}

__global__ void set_flag_kernel(int32_t *flag, int32_t v) { *flag = v; }

__global__ void check_symmetric_kernel(const uint16_t *__restrict__ s,
                                       const uint16_t *__restrict__ b, int64_t count,
                                       int32_t *__restrict__ result) {
  bool mismatch = false;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    float sc = __half2float(__ushort_as_half(s[i]));
    float bi = __half2float(__ushort_as_half(b[i]));
    // exact fp32 equality: +0 == -0, NaN != anything
    if (!(bi == __fmul_rn(-0.5f, sc))) mismatch = true;
  }
  if (__syncthreads_or(mismatch) && threadIdx.x == 0) *result = 0;
}

}  // namespace

cudaError_t launch_pack(const uint8_t *bits, int64_t N, int64_t K, uint32_t *w, cudaStream_t st) {
  int64_t nwords = N * (K / 32);
  pack_kernel<<<grid_for(nwords, 256), 256, 0, st>>>(bits, w, nwords);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t *w, int64_t N, int64_t K, uint8_t *bits,
                          cudaStream_t st) {
  int64_t nwords = N * (K / 32);
  unpack_kernel<<<grid_for(nwords, 256), 256, 0, st>>>(w, bits, nwords);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const WeightView &W, q1_dtype t, void *out, cudaStream_t st) {
  int64_t nwords = W.N * (W.K / 32);
  unsigned g = grid_for(nwords, 256);
  switch (t) {
    case Q1_BF16: dequantize_kernel<0><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, out); break;
    case Q1_F16: dequantize_kernel<1><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, out); break;
    default: dequantize_kernel<2><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, out); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_gather(const WeightView &E, const int32_t *ids, int64_t T, q1_dtype t,
                          void *out, int32_t *bad, cudaStream_t st) {
  int64_t nwords = T * (E.K / 32);
  unsigned g = grid_for(nwords, 256);
  switch (t) {
    case Q1_BF16:
      gather_kernel<0><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, ids, T, out, bad);
      break;
    case Q1_F16:
      gather_kernel<1><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, ids, T, out, bad);
      break;
    default:
      gather_kernel<2><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, ids, T, out, bad);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_check_symmetric(const WeightView &W, int32_t *result, cudaStream_t st) {
  set_flag_kernel<<<1, 1, 0, st>>>(result, 1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int64_t count = W.N * (W.K / 128);
  check_symmetric_kernel<<<grid_for(count, 256), 256, 0, st>>>(W.s, W.b, count, result);
  return cudaGetLastError();
}

}  // namespace q1
