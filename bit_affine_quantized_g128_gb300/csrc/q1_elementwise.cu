// Elementwise Q1 kernels: pack, unpack, dequantize, embedding gather, the
// symmetric-metadata check and the exact repack of dense tensors.  All of them are HBM-bound streams: one thread per
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

// The warp's 32 consecutive words: a lane's own word is word `lane` of the
// run starting at the warp's base.  The outputs of the run are contiguous, and
// every store instruction of the emitters below writes one contiguous 512
// bytes: store j puts chunk 32 j + lane (16 bytes) of the run, taking the word
// (and its values) from the lane that owns it.
constexpr unsigned kFull = 0xFFFFFFFFu;

__global__ void unpack_kernel(const uint32_t *__restrict__ w, uint8_t *__restrict__ bits,
                              int64_t nwords) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 32; base < nwords;
       base += nwarp * 32) {
    const bool valid = base + lane < nwords;
    const uint32_t v = valid ? w[base + lane] : 0u;
    const unsigned vmask = __ballot_sync(kFull, valid);
    uint4 *dst = reinterpret_cast<uint4 *>(bits + base * 32);
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // 32 bytes per word: 2 chunks of 16 bits
      const int c = 32 * j + lane, src = c >> 1;
      const uint32_t x = __shfl_sync(kFull, v, src) >> (16 * (c & 1));
      if ((vmask >> src) & 1u)
        dst[c] = make_uint4(nibble_to_bytes(x), nibble_to_bytes(x >> 4), nibble_to_bytes(x >> 8),
                            nibble_to_bytes(x >> 12));
    }
  }
}

// fp32 dequantized pair for one (row, group): lo = bias (q = 0),
// hi = fl32(scale + bias) (q = 1).  Symmetric: bias = -scale/2 in fp32 (exact).
__device__ __forceinline__ void group_values(const uint16_t *__restrict__ s,
                                             const uint16_t *__restrict__ b, int64_t idx, bool mbf16,
                                             float &lo, float &hi) {
  float sc = meta_f32(s[idx], mbf16);
  float bi = b ? meta_f32(b[idx], mbf16) : __fmul_rn(-0.5f, sc);
  lo = bi;
  hi = __fadd_rn(sc, bi);
}

// Output bit patterns of the dequantized pair (lo, hi) in the output dtype.
template <int OUT>  // 0 = bf16, 1 = f16, 2 = f32
__device__ __forceinline__ uint32_t out_bits(float v) {
  if (OUT == 2) return __float_as_uint(v);
  if (OUT == 0) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

// The warp's run of 32 words (lane: word `wd`, its values' patterns lo/hi,
// `valid` if inside the tensor) -> 32 x 32 outputs at `dst`, as contiguous
// 512-byte stores (see unpack_kernel).
template <int OUT>
__device__ __forceinline__ void warp_emit(uint32_t wd, uint32_t lo, uint32_t hi, bool valid, uint4 *dst) {
  constexpr int CPW = OUT == 2 ? 8 : 4;  // 16-byte chunks per word
  constexpr int VPC = 32 / CPW;          // values per chunk
  const int lane = threadIdx.x & 31;
  const unsigned vmask = __ballot_sync(kFull, valid);
#pragma unroll
  for (int j = 0; j < CPW; ++j) {
    const int c = 32 * j + lane, src = c / CPW;
    const uint32_t x = __shfl_sync(kFull, wd, src) >> (VPC * (c % CPW));
    const uint32_t l = __shfl_sync(kFull, lo, src), h = __shfl_sync(kFull, hi, src);
    if (!((vmask >> src) & 1u)) continue;
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (OUT == 2) q[e] = (x >> e) & 1u ? h : l;
      else q[e] = ((x >> (2 * e)) & 1u ? h : l) | (((x >> (2 * e + 1)) & 1u ? h : l) << 16);
    }
    dst[c] = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

template <int OUT>
__global__ void dequantize_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                                  const uint16_t *__restrict__ b, int64_t N, int64_t K, bool mbf16,
                                  int gshift, void *__restrict__ out) {
  const int64_t wpr = K / 32, G = wpr >> gshift, nwords = N * wpr;  // G: metadata groups per row
  const int esz = OUT == 2 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 32; base < nwords;
       base += nwarp * 32) {
    const int64_t i = base + lane;
    const bool valid = i < nwords;
    uint32_t wd = 0u, lo = 0u, hi = 0u;
    if (valid) {
      const int64_t n = i / wpr, c = i - n * wpr;
      float lf, hf;
      group_values(s, b, n * G + (c >> gshift), mbf16, lf, hf);
      wd = w[i];
      lo = out_bits<OUT>(lf);
      hi = out_bits<OUT>(hf);
    }
    // word i's 32 outputs start at element 32 i ([N][K] row-major, K = 32 wpr)
    warp_emit<OUT>(wd, lo, hi, valid, reinterpret_cast<uint4 *>(static_cast<char *>(out) + base * 32 * esz));
  }
}

template <int OUT>
__global__ void gather_kernel(const uint32_t *__restrict__ w, const uint16_t *__restrict__ s,
                              const uint16_t *__restrict__ b, int64_t V, int64_t K, bool mbf16,
                              int gshift, const int32_t *__restrict__ ids, int64_t T,
                              void *__restrict__ out, int32_t *__restrict__ bad) {
  const int64_t wpr = K / 32, G = wpr >> gshift, nwords = T * wpr;
  const int esz = OUT == 2 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 32; base < nwords;
       base += nwarp * 32) {
    const int64_t i = base + lane;
    const bool valid = i < nwords;
    uint32_t wd = 0u, lo = 0u, hi = 0u;  // an out-of-range id gives a zero row
    if (valid) {
      const int64_t t = i / wpr, c = i - t * wpr;
      const int64_t row = ids[t];
      if (row < 0 || row >= V) {
        if (c == 0 && bad) atomicAdd(bad, 1);
      } else {
        float lf, hf;
        group_values(s, b, row * G + (c >> gshift), mbf16, lf, hf);
        wd = w[row * wpr + c];
        lo = out_bits<OUT>(lf);
        hi = out_bits<OUT>(hf);
      }
    }
    // output word i (row t, word c) starts at element t K + 32 c = 32 i
    warp_emit<OUT>(wd, lo, hi, valid, reinterpret_cast<uint4 *>(static_cast<char *>(out) + base * 32 * esz));
  }
}

__global__ void set_flag_kernel(int32_t *flag, int32_t v) { *flag = v; }

// exact fp32 equality of a stored bias with -scale/2: +0 == -0, NaN != anything
__device__ __forceinline__ bool sym_pair(uint32_t sh, uint32_t bh, bool mbf16) {
  return meta_f32(bh, mbf16) == __fmul_rn(-0.5f, meta_f32(sh, mbf16));
}

// Eight groups per thread with 16-byte loads when both arrays are 16-byte
// aligned (vec), one group per thread otherwise.
__global__ void check_symmetric_kernel(const uint16_t *__restrict__ s,
                                       const uint16_t *__restrict__ b, int64_t count, bool mbf16,
                                       bool vec, int32_t *__restrict__ result) {
  bool mismatch = false;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t done = 0;
  if (vec) {
    const int64_t n8 = count / 8;
    const uint4 *s8 = reinterpret_cast<const uint4 *>(s), *b8 = reinterpret_cast<const uint4 *>(b);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += stride) {
      const uint4 sv = __ldg(s8 + i), bv = __ldg(b8 + i);
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (!sym_pair(sw[q], bw[q], mbf16) || !sym_pair(sw[q] >> 16, bw[q] >> 16, mbf16)) mismatch = true;
    }
    done = n8 * 8;
  }
  for (int64_t i = done + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count; i += stride)
    if (!sym_pair(s[i], b[i], mbf16)) mismatch = true;
  if (__syncthreads_or(mismatch) && threadIdx.x == 0) *result = 0;
}

// ---- exact repack from dense ("Bonsai masked gemv", cactus PR #775: tensors
// whose 128-groups hold exactly two values repack with zero quantization error;
// anything else is refused).  One warp per group; lane l holds the group's
// values 4l .. 4l+3 as fp32 bit patterns (bf16 and fp16 widen exactly, so
// patterns compare like the input's).

// One fp16 step along the number line (nextafter toward +inf or -inf) of a
// finite fp16 bit pattern.
__device__ __forceinline__ uint32_t f16_next(uint32_t h, bool up) {
  if ((h & 0x7FFFu) == 0u) return up ? 0x0001u : 0x8001u;  // from +-0 to +-(smallest subnormal)
  const bool neg = (h & 0x8000u) != 0u;
  return (up != neg) ? h + 1u : h - 1u;
}

// The fp32 bit patterns of lane l's values 4l .. 4l+3 of the group at element e0.
template <int DT>
__device__ __forceinline__ void load_group(const void *__restrict__ dense, int64_t e0, uint32_t (&p)[4]) {
  if (DT == 2) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(dense) + e0));
    p[0] = v.x; p[1] = v.y; p[2] = v.z; p[3] = v.w;
  } else {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(dense) + e0));
    p[0] = v.x & 0xFFFFu; p[1] = v.x >> 16; p[2] = v.y & 0xFFFFu; p[3] = v.y >> 16;
  }
}

template <int DT>
__device__ __forceinline__ void widen(uint32_t (&p)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (DT == 0) p[j] <<= 16;
    if (DT == 1) p[j] = __float_as_uint(__half2float(__ushort_as_half((uint16_t)p[j])));
  }
}

// The metadata of one group from its values A and B (B == A: one value):
// scale, bias, the pattern whose weights get bit 1 (two values) or whether
// all bits are 1 (one value); false when the group is refused.
__device__ __forceinline__ bool group_meta(uint32_t A, uint32_t B, bool two, bool ok, int symmetric,
                                           uint32_t &hi_pat, bool &allone, uint32_t &sc, uint32_t &bi) {
  hi_pat = 0u;
  allone = false;
  sc = 0u;
  bi = 0u;
  if (ok && !two) {
    const float x = __uint_as_float(A);
    if (symmetric) {
      const bool neg = (A >> 31) != 0u;
      sc = __half_as_ushort(__float2half_rn(__fmul_rn(neg ? -2.0f : 2.0f, x)));
      const float sf = __half2float(__ushort_as_half((uint16_t)sc));
      const float bb = __fmul_rn(-0.5f, sf);
      ok = __float_as_uint(neg ? bb : __fadd_rn(sf, bb)) == A;
      allone = !neg;
    } else {
      bi = __half_as_ushort(__float2half_rn(x));
      ok = __float_as_uint(__half2float(__ushort_as_half((uint16_t)bi))) == A;
    }
  } else if (ok) {
    const float fa = __uint_as_float(A), fb = __uint_as_float(B);
    const bool a_lo = fa < fb || (fa == fb && (A >> 31) != 0u);  // -0 below +0
    const uint32_t lo_pat = a_lo ? A : B;
    hi_pat = a_lo ? B : A;
    const float lo = __uint_as_float(lo_pat), hi = __uint_as_float(hi_pat);
    if (symmetric) {
      sc = __half_as_ushort(__float2half_rn(__fmul_rn(-2.0f, lo)));
      const float sf = __half2float(__ushort_as_half((uint16_t)sc));
      const float bb = __fmul_rn(-0.5f, sf);
      ok = __float_as_uint(bb) == lo_pat && __float_as_uint(__fadd_rn(sf, bb)) == hi_pat;
    } else {
      bi = __half_as_ushort(__float2half_rn(lo));
      const float bf = __half2float(__ushort_as_half((uint16_t)bi));
      ok = __float_as_uint(bf) == lo_pat;
      if (ok) {
        // scales tried: RN16(hi - lo), then one step down, one up, two down, two up
        const uint32_t c0 = __half_as_ushort(__float2half_rn(__fsub_rn(hi, lo)));
        const uint32_t dn1 = f16_next(c0, false), up1 = f16_next(c0, true);
        const uint32_t cands[5] = {c0, dn1, up1, f16_next(dn1, false), f16_next(up1, true)};
        ok = false;
#pragma unroll
        for (int t = 0; t < 5; ++t) {
          if (ok || (cands[t] & 0x7C00u) == 0x7C00u) continue;
          const float sf = __half2float(__ushort_as_half((uint16_t)cands[t]));
          if (__float_as_uint(__fadd_rn(sf, bf)) == hi_pat) {
            ok = true;
            sc = cands[t];
          }
        }
      }
    }
  }
  if (!ok) {
    sc = 0u;
    bi = 0u;
  }
  return ok;
}

// One warp per run of kRepackRun consecutive groups.  All the run's loads are
// issued first (bytes in flight); then, per group, the warp finds its values
// (lane 0's first value A; B = the first value that differs, by ballot; a
// vote refuses a third); then lane u works out the metadata of group u of the
// run, once; then each group's decisions are broadcast and its bits packed.
constexpr int kRepackRun = 8;

template <int DT>  // input: 0 bf16, 1 fp16, 2 fp32
__global__ void pack_from_dense_kernel(const void *__restrict__ dense, int64_t N, int64_t K,
                                       int symmetric, uint32_t *__restrict__ w,
                                       uint16_t *__restrict__ s, uint16_t *__restrict__ b,
                                       int32_t *__restrict__ bad) {
  const unsigned FULL = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  const int me = lane & (kRepackRun - 1);
  const int64_t ngroups = N * (K / 128);
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t grp0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kRepackRun; grp0 < ngroups;
       grp0 += nw * kRepackRun) {
    // groups are numbered row-major (n * G + g), so a run is contiguous in
    // memory: group grp starts at element grp * 128
    uint32_t p[kRepackRun][4];
#pragma unroll
    for (int u = 0; u < kRepackRun; ++u) {
      if (grp0 + u < ngroups) load_group<DT>(dense, (grp0 + u) * 128 + 4 * lane, p[u]);
      else p[u][0] = p[u][1] = p[u][2] = p[u][3] = 0u;
    }
    // per group: the values A, B and the vote
    uint32_t mA = 0u, mB = 0u;
    bool mtwo = false, mok = false;
#pragma unroll
    for (int u = 0; u < kRepackRun; ++u) {
      widen<DT>(p[u]);
      const uint32_t A = __shfl_sync(FULL, p[u][0], 0);
      uint32_t cand = A;
      bool has = false;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (!has && p[u][j] != A) { cand = p[u][j]; has = true; }
      const uint32_t hb = __ballot_sync(FULL, has);
      const uint32_t B = hb ? __shfl_sync(FULL, cand, __ffs(hb) - 1) : A;
      bool viol = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) viol |= p[u][j] != A && p[u][j] != B;
      const bool finite = (A & 0x7F800000u) != 0x7F800000u && (B & 0x7F800000u) != 0x7F800000u;
      const bool ok = !__any_sync(FULL, viol) && finite;
      if (me == u) {
        mA = A;
        mB = B;
        mtwo = hb != 0u;
        mok = ok;
      }
    }
    // lane u (and its copies u + 8, u + 16, u + 24): group u's metadata
    uint32_t hi_pat, sc, bi;
    bool allone;
    const bool ok = group_meta(mA, mB, mtwo, mok, symmetric, hi_pat, allone, sc, bi);
    const int64_t my = grp0 + me;
    if (lane < kRepackRun && my < ngroups) {
      s[my] = (uint16_t)sc;
      if (b) b[my] = (uint16_t)bi;
      if (!ok) atomicAdd(bad, 1);
    }
    // the bits: weights equal to hi (two values) or the single value's rule;
    // word l / 8 of a group takes lane l's nibble at bits 4 (l % 8) .. +3
#pragma unroll
    for (int u = 0; u < kRepackRun; ++u) {
      const int64_t grp = grp0 + u;
      if (grp >= ngroups) break;  // uniform across the warp
      const uint32_t hp = __shfl_sync(FULL, hi_pat, u);
      const int mode = __shfl_sync(FULL, ok ? (mtwo ? 2 : (allone ? 1 : 0)) : 0, u);
      uint32_t nib = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool bit = mode == 2 ? p[u][j] == hp : mode == 1;
        nib |= (bit ? 1u : 0u) << j;
      }
      uint32_t word = nib << (4 * (lane & 7));
      word |= __shfl_xor_sync(FULL, word, 1);
      word |= __shfl_xor_sync(FULL, word, 2);
      word |= __shfl_xor_sync(FULL, word, 4);
      if ((lane & 7) == 0) w[grp * 4 + (lane >> 3)] = word;
    }
  }
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
  unpack_kernel<<<grid_for((nwords + 31) / 32 * 32, 256), 256, 0, st>>>(w, bits, nwords);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const WeightView &W, q1_dtype t, void *out, cudaStream_t st) {
  int64_t nwords = W.N * (W.K / 32);
  unsigned g = grid_for(nwords, 256);
  switch (t) {
    case Q1_BF16: dequantize_kernel<0><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, W.mbf16, W.gshift, out); break;
    case Q1_F16: dequantize_kernel<1><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, W.mbf16, W.gshift, out); break;
    default: dequantize_kernel<2><<<g, 256, 0, st>>>(W.w, W.s, W.b, W.N, W.K, W.mbf16, W.gshift, out); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_gather(const WeightView &E, const int32_t *ids, int64_t T, q1_dtype t,
                          void *out, int32_t *bad, cudaStream_t st) {
  int64_t nwords = T * (E.K / 32);
  unsigned g = grid_for(nwords, 256);
  switch (t) {
    case Q1_BF16:
      gather_kernel<0><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, E.mbf16, E.gshift, ids, T, out, bad);
      break;
    case Q1_F16:
      gather_kernel<1><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, E.mbf16, E.gshift, ids, T, out, bad);
      break;
    default:
      gather_kernel<2><<<g, 256, 0, st>>>(E.w, E.s, E.b, E.N, E.K, E.mbf16, E.gshift, ids, T, out, bad);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_check_symmetric(const WeightView &W, int32_t *result, cudaStream_t st) {
  set_flag_kernel<<<1, 1, 0, st>>>(result, 1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  int64_t count = W.N * ((W.K / 32) >> W.gshift);
  const bool vec = (reinterpret_cast<uintptr_t>(W.s) & 15) == 0 && (reinterpret_cast<uintptr_t>(W.b) & 15) == 0;
  check_symmetric_kernel<<<grid_for(vec ? count / 8 + 1 : count, 256), 256, 0, st>>>(W.s, W.b, count, W.mbf16, vec,
                                                                                   result);
  return cudaGetLastError();
}

cudaError_t launch_pack_from_dense(const void *dense, q1_dtype t, int64_t N, int64_t K, uint32_t *w,
                                   uint16_t *s, uint16_t *b, int32_t *bad, cudaStream_t st) {
  const int64_t groups = N * (K / 128);
  const unsigned g = grid_for((groups + kRepackRun - 1) / kRepackRun * 32, 256);
  const int sym = b == nullptr ? 1 : 0;
  switch (t) {
    case Q1_BF16: pack_from_dense_kernel<0><<<g, 256, 0, st>>>(dense, N, K, sym, w, s, b, bad); break;
    case Q1_F16: pack_from_dense_kernel<1><<<g, 256, 0, st>>>(dense, N, K, sym, w, s, b, bad); break;
    default: pack_from_dense_kernel<2><<<g, 256, 0, st>>>(dense, N, K, sym, w, s, b, bad); break;
  }
  return cudaGetLastError();
}

}  // namespace q1
