// Internal declarations shared by the library's translation units (host side).
// Not part of the public ABI (include/q1.h is).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "q1.h"

namespace q1 {

// One-time host state is kept per device: a process may drive several GPUs,
// and function attributes, SM counts and occupancy are per device.  Devices
// beyond kMaxDevices are served without caching.
constexpr int kMaxDevices = 64;
inline int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0) d = 0;
  return d;
}
// True once per (flag, device): the caller then does the one-time work and,
// if it succeeded, calls mark_done.  Concurrent first calls may both do it.
inline bool not_done(const std::atomic<uint64_t> &flag, int dev) {
  return dev >= kMaxDevices || !(flag.load(std::memory_order_relaxed) & (1ull << dev));
}
inline void mark_done(std::atomic<uint64_t> &flag, int dev) {
  if (dev < kMaxDevices) flag.fetch_or(1ull << dev, std::memory_order_relaxed);
}

constexpr int kGroup = 128;      // weights per scale/bias group
constexpr int kWordBits = 32;    // weights per packed word
constexpr int kNarrowMaxM = 8;   // token rows of one mma.sync n8 tile
// K of the narrow kernel: a cluster of at most 8 CTAs x 10 span warps x 512 k
constexpr int64_t kNarrowMaxK = 8 * 10 * 512;

// Metadata pointers resolved for a launch.
struct WeightView {
  const uint32_t *w;
  const uint16_t *s;
  const uint16_t *b;  // nullptr: symmetric
  int64_t N, K;
  bool mbf16;         // scales/biases are bf16 (else fp16)
  int gshift;         // log2(group_size / 32): 0, 1 or 2
};

inline WeightView view(const q1_weight *W) {
  return WeightView{W->w, W->scales, W->biases, W->N, W->K, W->meta_dtype == Q1_META_BF16,
                    W->group_size == 32 ? 0 : (W->group_size == 64 ? 1 : 2)};
}

#ifdef __CUDACC__
// One fp16 or bf16 metadata value (its 16 bits in the low half of h) -> fp32;
// both widenings are exact.
__device__ __forceinline__ float meta_f32(uint32_t h, bool bf16) {
  return bf16 ? __uint_as_float((h & 0xFFFFu) << 16) : __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}
#endif

// ---- elementwise kernels (q1_elementwise.cu)
cudaError_t launch_pack(const uint8_t *bits, int64_t N, int64_t K, uint32_t *w, cudaStream_t st);
cudaError_t launch_unpack(const uint32_t *w, int64_t N, int64_t K, uint8_t *bits,
                          cudaStream_t st);
cudaError_t launch_dequantize(const WeightView &W, q1_dtype t, void *out, cudaStream_t st);
cudaError_t launch_gather(const WeightView &E, const int32_t *ids, int64_t T, q1_dtype t,
                          void *out, int32_t *bad, cudaStream_t st);
cudaError_t launch_check_symmetric(const WeightView &W, int32_t *result, cudaStream_t st);
// w/s/b [N][K/32], [N][K/128]: the exact Q1 form of dense [N][K] (b == nullptr:
// symmetric); refused groups are zeroed and counted in *bad.
cudaError_t launch_pack_from_dense(const void *dense, q1_dtype t, int64_t N, int64_t K, uint32_t *w,
                                   uint16_t *s, uint16_t *b, int32_t *bad, cudaStream_t st);

// ---- narrow path (q1_narrow.cu): one launch, no scratch
// y [M][N] (ydt) = x . W^T (x [M][K], xdt); fp16/fp32 x are rounded to bf16,
// the tensor-core operand type, as they are loaded.
cudaError_t launch_narrow(const WeightView &W, const void *x, int64_t M, void *y,
                          cudaStream_t st, bool pdl, q1_dtype xdt = Q1_BF16, q1_dtype ydt = Q1_BF16);
// h [M][F] bf16 = SiLU(x . G^T) * (x . U^T), x in xdt.
cudaError_t launch_narrow_gate_up(const WeightView &G, const WeightView &U, const void *x,
                                  int64_t M, void *h, cudaStream_t st, bool pdl, q1_dtype xdt = Q1_BF16);

// ---- wide path (q1_wide.cu)
// workspace: fp16 activation rows [M][K], per-row scales [M] and, when the
// launch plan for this shape shares tiles between CTA pairs, partial-sum slots
// and share counts
size_t wide_workspace_bytes(int64_t M, int64_t N, int64_t K);
// x [M][K] and y [M][N] in dt (bf16, fp16 or fp32); ws of ws_bytes >= wide_workspace_bytes
cudaError_t launch_wide(const WeightView &W, const void *x, int64_t M, void *y, void *ws, size_t ws_bytes,
                        cudaStream_t st, q1_dtype dt = Q1_BF16);
// fixed prefill tiling (token_tile, split), or the automatic choice when invalid
void set_pair_plan(int token_tile, int split);

// ---- device error words (each translation unit with bounded waits owns one)
// and the diagnostics of the bounded waits: their limit, and producers that
// issue nothing (every wait for their data then runs out)
cudaError_t set_narrow_diagnostics(unsigned long long wait_ns, int stall);
cudaError_t set_wide_diagnostics(unsigned long long wait_ns, int stall);
unsigned int read_and_clear_wide_errors(cudaStream_t st, cudaError_t *err);
unsigned int read_and_clear_narrow_errors(cudaStream_t st, cudaError_t *err);

}  // namespace q1
