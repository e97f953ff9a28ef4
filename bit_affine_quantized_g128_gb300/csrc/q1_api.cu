// C ABI entry points of libq1 (declared in include/q1.h): host-side argument
// validation, dispatch between the narrow and wide matmul paths, and launch
// chaining.  No device memory is allocated here; scratch (the prefill path's
// fp16 activation rows, the fused FFN's intermediate) comes from the caller's
// workspace.
#include <atomic>
#include <cstdlib>
#include <cstring>

#include "q1_internal.h"

namespace {

using q1::WeightView;

std::atomic<int> g_max_rows{[] {
  const char *e = std::getenv("Q1_QMM_MAX_ROWS");
  if (!e) return 8;
  int v = std::atoi(e);
  return v < 0 ? 0 : (v > 8 ? 8 : v);
}()};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

q1_status cuda_status(cudaError_t e) { return e == cudaSuccess ? Q1_OK : Q1_ERR_CUDA; }

// The kernels use tcgen05 / sm_103a features: refuse other devices loudly.
q1_status check_device() {
  static thread_local int checked_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q1_ERR_CUDA;
  if (dev == checked_dev) return Q1_OK;
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return Q1_ERR_CUDA;
  if (major != 10) return Q1_ERR_DEVICE;
  checked_dev = dev;
  return Q1_OK;
}

q1_status check_weight(const q1_weight *W) {
  if (!W || !W->w || !W->scales) return Q1_ERR_NULL;
  if (W->group_size != 32 && W->group_size != 64 && W->group_size != 128) return Q1_ERR_GROUP;
  if (W->meta_dtype != Q1_META_F16 && W->meta_dtype != Q1_META_BF16) return Q1_ERR_DTYPE;
  if (W->N < 1 || W->K < 128 || W->K % 128 != 0) return Q1_ERR_SHAPE;
  if (W->K > (int64_t)1 << 24 || W->N > ((int64_t)1 << 31) - 1) return Q1_ERR_SHAPE;
  if (!aligned(W->w, 16) || !aligned(W->scales, 2) || (W->biases && !aligned(W->biases, 2)))
    return Q1_ERR_ALIGN;
  return Q1_OK;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

q1_status check_ws(const void *ws, size_t have, size_t need) {
  if (need == 0) return Q1_OK;
  if (!ws) return Q1_ERR_WORKSPACE;
  if (have < need || !aligned(ws, 256)) return Q1_ERR_WORKSPACE;
  return Q1_OK;
}

q1_status matmul_common(const q1_weight *W, const void *x, int64_t M, q1_dtype dtype,
                        const void *y) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  s = check_weight(W);
  if (s != Q1_OK) return s;
  if (!x || !y) return Q1_ERR_NULL;
  if (dtype != Q1_BF16 && dtype != Q1_F16 && dtype != Q1_F32) return Q1_ERR_DTYPE;
  if (M < 1 || M > ((int64_t)1 << 24)) return Q1_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 16)) return Q1_ERR_ALIGN;
  return Q1_OK;
}

}  // namespace

extern "C" {

const char *q1_status_string(q1_status s) {
  switch (s) {
    case Q1_OK: return "ok";
    case Q1_ERR_NULL: return "a required pointer is NULL";
    case Q1_ERR_SHAPE: return "invalid shape (need N>=1, K>=128, K%128==0, M in range)";
    case Q1_ERR_ALIGN: return "pointer misaligned (packed words, x, y, out: 16 bytes)";
    case Q1_ERR_DTYPE: return "unsupported dtype for this call";
    case Q1_ERR_GROUP: return "group_size must be 32, 64 or 128 (gate and up of one FFN: the same)";
    case Q1_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case Q1_ERR_CUDA: return "CUDA runtime error";
    case Q1_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case Q1_ERR_DEVICE: return "current device is not a compute capability 10.x (Blackwell) GPU";
  }
  return "unknown status";
}

void q1_set_qmm_max_rows(int rows) { g_max_rows.store(rows < 0 ? 0 : (rows > 8 ? 8 : rows)); }
int q1_get_qmm_max_rows(void) { return g_max_rows.load(); }
void q1_set_prefill_plan(int token_tile, int split) { q1::set_pair_plan(token_tile, split); }

q1_status q1_pack(const uint8_t *bits, int64_t N, int64_t K, uint32_t *w, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  if (!bits || !w) return Q1_ERR_NULL;
  if (N < 1 || K < 32 || K % 32 != 0) return Q1_ERR_SHAPE;
  if (!aligned(bits, 16) || !aligned(w, 16)) return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_pack(bits, N, K, w, (cudaStream_t)stream));
}

q1_status q1_unpack(const uint32_t *w, int64_t N, int64_t K, uint8_t *bits, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  if (!bits || !w) return Q1_ERR_NULL;
  if (N < 1 || K < 32 || K % 32 != 0) return Q1_ERR_SHAPE;
  if (!aligned(bits, 16) || !aligned(w, 16)) return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_unpack(w, N, K, bits, (cudaStream_t)stream));
}

q1_status q1_dequantize(const q1_weight *W, q1_dtype out_t, void *out, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  s = check_weight(W);
  if (s != Q1_OK) return s;
  if (!out) return Q1_ERR_NULL;
  if (out_t != Q1_BF16 && out_t != Q1_F16 && out_t != Q1_F32) return Q1_ERR_DTYPE;
  if (!aligned(out, 16)) return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_dequantize(q1::view(W), out_t, out, (cudaStream_t)stream));
}

q1_status q1_qmv(const q1_weight *W, const void *x, q1_dtype dtype, void *y, q1_stream stream) {
  q1_status s = matmul_common(W, x, 1, dtype, y);
  if (s != Q1_OK) return s;
  if (W->K > q1::kNarrowMaxK) return Q1_ERR_SHAPE;
  return cuda_status(q1::launch_narrow(q1::view(W), x, 1, y, (cudaStream_t)stream, true, dtype, dtype));
}

q1_status q1_qmm_narrow(const q1_weight *W, const void *x, int64_t M, q1_dtype dtype, void *y,
                        q1_stream stream) {
  q1_status s = matmul_common(W, x, M, dtype, y);
  if (s != Q1_OK) return s;
  if (M > q1::kNarrowMaxM || W->K > q1::kNarrowMaxK) return Q1_ERR_SHAPE;
  return cuda_status(q1::launch_narrow(q1::view(W), x, M, y, (cudaStream_t)stream, true, dtype, dtype));
}

size_t q1_qmm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || K < 128 || K % 128) return 0;
  return q1::wide_workspace_bytes(M, N, K);
}

q1_status q1_qmm(const q1_weight *W, const void *x, int64_t M, q1_dtype dtype, void *y,
                 void *workspace, size_t workspace_bytes, q1_stream stream) {
  q1_status s = matmul_common(W, x, M, dtype, y);
  if (s != Q1_OK) return s;
  const int rows = g_max_rows.load();
  if (M <= rows && W->K <= q1::kNarrowMaxK)
    return cuda_status(q1::launch_narrow(q1::view(W), x, M, y, (cudaStream_t)stream, true, dtype, dtype));
  if (rows == q1::kNarrowMaxM && M <= 2 * q1::kNarrowMaxM && W->K <= q1::kNarrowMaxK) {
    // 9..16 rows at the default threshold: two narrow launches of 8 rows and
    // M - 8 rows, the second chained with PDL (it streams its weights while
    // the first drains).  Twice the weight traffic costs less than the
    // prefill path here, whose MMAs take as long for 16 tokens as for 256.
    const size_t es = dtype == Q1_F32 ? 4 : 2;
    const int64_t m0 = q1::kNarrowMaxM;
    cudaError_t e = q1::launch_narrow(q1::view(W), x, m0, y, (cudaStream_t)stream, true, dtype, dtype);
    if (e == cudaSuccess)
      e = q1::launch_narrow(q1::view(W), static_cast<const char *>(x) + (size_t)m0 * W->K * es, M - m0,
                            static_cast<char *>(y) + (size_t)m0 * W->N * es, (cudaStream_t)stream, true, dtype,
                            dtype);
    return cuda_status(e);
  }
  s = check_ws(workspace, workspace_bytes, q1::wide_workspace_bytes(M, W->N, W->K));
  if (s != Q1_OK) return s;
  return cuda_status(q1::launch_wide(q1::view(W), x, M, y, workspace, workspace_bytes, (cudaStream_t)stream, dtype));
}

q1_status q1_embed_gather(const q1_weight *E, const int32_t *ids, int64_t T, q1_dtype out_t,
                          void *out, int32_t *d_bad_count, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  s = check_weight(E);
  if (s != Q1_OK) return s;
  if (T < 0) return Q1_ERR_SHAPE;
  if (T == 0) return Q1_OK;
  if (!ids || !out) return Q1_ERR_NULL;
  if (out_t != Q1_BF16 && out_t != Q1_F16 && out_t != Q1_F32) return Q1_ERR_DTYPE;
  if (!aligned(out, 16) || !aligned(ids, 4) || (d_bad_count && !aligned(d_bad_count, 4)))
    return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_gather(q1::view(E), ids, T, out_t, out, d_bad_count,
                                       (cudaStream_t)stream));
}

size_t q1_ffn_workspace_size(int64_t M, int64_t D, int64_t F) {
  if (M < 1 || M > 8 || D < 128 || F < 128 || D % 128 || F % 128) return 0;
  return align256((size_t)(M * F * 2));  // h [M][F] bf16
}

q1_status q1_ffn_fused(const q1_weight *gate, const q1_weight *up, const q1_weight *down,
                       const void *x, int64_t M, q1_dtype dtype, void *y, void *workspace,
                       size_t workspace_bytes, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  if ((s = check_weight(gate)) != Q1_OK || (s = check_weight(up)) != Q1_OK ||
      (s = check_weight(down)) != Q1_OK)
    return s;
  // gate and up run in one launch with one group size; down may differ
  if (gate->group_size != up->group_size) return Q1_ERR_GROUP;
  if (!x || !y) return Q1_ERR_NULL;
  if (dtype != Q1_BF16 && dtype != Q1_F16 && dtype != Q1_F32) return Q1_ERR_DTYPE;
  if (M < 1 || M > q1::kNarrowMaxM) return Q1_ERR_SHAPE;
  const int64_t D = gate->K, F = gate->N;
  if (up->K != D || up->N != F || down->K != F || down->N != D) return Q1_ERR_SHAPE;
  if (D > q1::kNarrowMaxK || F > q1::kNarrowMaxK) return Q1_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(y, 16)) return Q1_ERR_ALIGN;
  s = check_ws(workspace, workspace_bytes, q1_ffn_workspace_size(M, D, F));
  if (s != Q1_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  void *h = workspace;
  // two launches chained with programmatic dependent launch: the down
  // projection starts streaming its weights while gate/up drains, and waits
  // for h only before reading it
  cudaError_t e = q1::launch_narrow_gate_up(q1::view(gate), q1::view(up), x, M, h, st, true, dtype);
  if (e == cudaSuccess) e = q1::launch_narrow(q1::view(down), h, M, y, st, true, Q1_BF16, dtype);
  return cuda_status(e);
}

size_t q1_decode_chain_workspace_size(int64_t M, int64_t D, int64_t F_max) {
  if (M < 1 || M > 8 || D < 128 || F_max < 128 || D % 128 || F_max % 128) return 0;
  // a [M][D], the current h [M][D], the FFN intermediate [M][F_max], all bf16
  return 2 * align256((size_t)(M * D * 2)) + align256((size_t)(M * F_max * 2));
}

q1_status q1_decode_chain(const q1_decode_layer *layers, int32_t n_layers, const void *x,
                          int64_t M, q1_dtype dtype, void *y, void *workspace,
                          size_t workspace_bytes, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  if (!layers || !x || !y) return Q1_ERR_NULL;
  if (n_layers < 1) return Q1_ERR_SHAPE;
  if (dtype != Q1_BF16) return Q1_ERR_DTYPE;
  if (M < 1 || M > q1::kNarrowMaxM) return Q1_ERR_SHAPE;
  const int64_t D = layers[0].attn.N;
  int64_t F_max = 0;
  for (int32_t l = 0; l < n_layers; ++l) {
    const q1_decode_layer &L = layers[l];
    if ((s = check_weight(&L.attn)) != Q1_OK || (s = check_weight(&L.gate)) != Q1_OK ||
        (s = check_weight(&L.up)) != Q1_OK || (s = check_weight(&L.down)) != Q1_OK)
      return s;
    if (L.gate.group_size != L.up.group_size) return Q1_ERR_GROUP;
    const int64_t F = L.gate.N;
    if (L.attn.N != D || L.attn.K != D || L.gate.K != D || L.up.K != D || L.up.N != F ||
        L.down.K != F || L.down.N != D)
      return Q1_ERR_SHAPE;
    if (D > q1::kNarrowMaxK || F > q1::kNarrowMaxK) return Q1_ERR_SHAPE;
    F_max = F > F_max ? F : F_max;
  }
  if (!aligned(x, 16) || !aligned(y, 16)) return Q1_ERR_ALIGN;
  s = check_ws(workspace, workspace_bytes, q1_decode_chain_workspace_size(M, D, F_max));
  if (s != Q1_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  char *ws = static_cast<char *>(workspace);
  void *a = ws;
  void *hb = ws + align256((size_t)(M * D * 2));
  void *fh = ws + 2 * align256((size_t)(M * D * 2));
  cudaError_t e = cudaSuccess;
  for (int32_t l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const q1_decode_layer &L = layers[l];
    const void *in = l == 0 ? x : hb;
    void *out = l == n_layers - 1 ? y : hb;
    // every kernel reads its input only after its predecessor has completed
    // (griddepcontrol.wait), and each predecessor completed only after its own
    // predecessor: the down projection overwrites hb after the attention
    // product that read it is done
    e = q1::launch_narrow(q1::view(&L.attn), in, M, a, st, true);
    if (e == cudaSuccess) e = q1::launch_narrow_gate_up(q1::view(&L.gate), q1::view(&L.up), a, M, fh, st, true);
    if (e == cudaSuccess) e = q1::launch_narrow(q1::view(&L.down), fh, M, out, st, true);
  }
  return cuda_status(e);
}

q1_status q1_pack_from_dense(const void *dense, q1_dtype in_t, int64_t N, int64_t K, uint32_t *w,
                             uint16_t *scales, uint16_t *biases, int32_t *d_bad_groups,
                             q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  if (!dense || !w || !scales || !d_bad_groups) return Q1_ERR_NULL;
  if (in_t != Q1_BF16 && in_t != Q1_F16 && in_t != Q1_F32) return Q1_ERR_DTYPE;
  if (N < 1 || K < 128 || K % 128 != 0 || K > (int64_t)1 << 24 || N > ((int64_t)1 << 31) - 1)
    return Q1_ERR_SHAPE;
  if (!aligned(dense, 16) || !aligned(w, 16) || !aligned(scales, 2) || (biases && !aligned(biases, 2)) ||
      !aligned(d_bad_groups, 4))
    return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_pack_from_dense(dense, in_t, N, K, w, scales, biases, d_bad_groups,
                                                (cudaStream_t)stream));
}

q1_status q1_check_symmetric(const q1_weight *W, int32_t *d_is_symmetric, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  s = check_weight(W);
  if (s != Q1_OK) return s;
  if (!W->biases || !d_is_symmetric) return Q1_ERR_NULL;
  if (!aligned(d_is_symmetric, 4)) return Q1_ERR_ALIGN;
  return cuda_status(q1::launch_check_symmetric(q1::view(W), d_is_symmetric, (cudaStream_t)stream));
}

namespace {
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_stall{0};
q1_status push_diagnostics() {
  const unsigned long long ns = g_wait_ns.load();
  const int stall = g_stall.load();
  cudaError_t e = q1::set_narrow_diagnostics(ns, stall);
  if (e == cudaSuccess) e = q1::set_wide_diagnostics(ns, stall);
  return cuda_status(e);
}
}  // namespace

q1_status q1_set_wait_limit_ns(uint64_t ns) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  g_wait_ns.store(ns ? (unsigned long long)ns : 2000000000ull);
  return push_diagnostics();
}

q1_status q1_set_stalled_producers(int stall) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  g_stall.store(stall ? 1 : 0);
  return push_diagnostics();
}

q1_status q1_device_errors(unsigned int *flags, q1_stream stream) {
  q1_status s = check_device();
  if (s != Q1_OK) return s;
  cudaError_t e1 = cudaSuccess, e2 = cudaSuccess;
  unsigned int v = q1::read_and_clear_wide_errors((cudaStream_t)stream, &e1);
  v |= q1::read_and_clear_narrow_errors((cudaStream_t)stream, &e2) << 1;
  if (flags) *flags = v;
  if (e1 != cudaSuccess || e2 != cudaSuccess) return Q1_ERR_CUDA;
  return v ? Q1_ERR_TIMEOUT : Q1_OK;
}

}  // extern "C"
