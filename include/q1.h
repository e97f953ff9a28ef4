/*
 * q1.h - C ABI of libq1: the 1-bit affine group-quantized (group size 128)
 * linear layer on NVIDIA GB300 (sm_103a).
 *
 * Format ("1-bit affine weight support", rMLX issue #207, section "The good
 * news - packing is standard"; "Bonsai masked gemv", cactus PR #775, "linear
 * LSB layout"):
 *   w       uint32 [N][K/32]  weight (n, k) is bit (k % 32) of word [n][k / 32]
 *   scales  fp16   [N][K/128] one per row and group of 128 along K
 *   biases  fp16   [N][K/128] or NULL
 *   (bf16 metadata and group sizes 32 / 64 are variants: see q1_weight)
 * Value ("Support Bonsai-27B affine Q1", higgs PR #212, section "What"):
 *   w(n,k) = scale * q + bias, q in {0,1}.  With biases == NULL the tensor is
 *   symmetric: bias = -scale/2, derived in fp32 and never stored.  So bit 0
 *   gives the negative value and bit 1 the positive one.
 *   The dequantized value is fp32: q = 0 -> bias, q = 1 -> fl32(scale + bias).
 *
 * Conventions for every call:
 *   - Pointers named d_* or documented as "device" are device pointers
 *     allocated by the caller (the library never allocates or frees device
 *     memory).  Arrays are row-major and contiguous.  The library cannot tell
 *     a host pointer, or an output array shorter than the call writes, from a
 *     good one: passing either is undefined behaviour (the Python binding
 *     checks both before it calls in).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *     call returns without waiting, unless stated otherwise.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid argument returns an error status and launches nothing.  A failed
 *     launch returns Q1_ERR_CUDA.  No exception crosses the ABI.
 *   - Activations and outputs of the matmul and FFN calls share one dtype:
 *     Q1_BF16, Q1_F16 or Q1_F32 (q1_decode_chain: Q1_BF16 only).  The narrow
 *     path's tensor-core operands are bf16, so fp16 and fp32 activations are
 *     rounded once to bf16 as they are loaded (relative error <= 2^-9 per
 *     activation); the prefill path scales them into fp16 rows (exact for bf16
 *     and fp16 activations, one rounding at 2^-11 for fp32).  Accumulation is
 *     fp32 and the output is rounded once to the dtype.
 *   - Calls that need scratch (q1_qmm on its prefill path, q1_ffn_fused and
 *     q1_decode_chain for their intermediate activations) take a caller-owned
 *     device workspace and its size; q1_qmm_workspace_size,
 *     q1_ffn_workspace_size and q1_decode_chain_workspace_size return the
 *     bytes needed.  A workspace must be 256-byte aligned and must not be used
 *     by another call that may run concurrently.
 *   - Device-side waits in the kernels are bounded; one that runs out sets a
 *     device error word that q1_device_errors() reads (Q1_ERR_TIMEOUT).
 *   - The narrow matmul and FFN kernels are launched with programmatic
 *     dependent launch: they may start streaming the packed weights and
 *     metadata while the preceding kernel on the stream is still running, if
 *     that kernel signalled programmatic completion early; they read x (and
 *     write y) only after the preceding kernel has completed.  Weights must
 *     therefore not be produced by a kernel that signals early.
 */
#ifndef Q1_H_
#define Q1_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *q1_stream;

typedef enum {
  Q1_OK = 0,
  Q1_ERR_NULL = 1,       /* a required pointer is NULL                          */
  Q1_ERR_SHAPE = 2,      /* N < 1, K < 128, K % 128 != 0, M out of range, ...   */
  Q1_ERR_ALIGN = 3,      /* a pointer is not aligned as documented              */
  Q1_ERR_DTYPE = 4,      /* unsupported dtype for this call                     */
  Q1_ERR_GROUP = 5,      /* group_size not 32, 64 or 128, or not 128 where needed */
  Q1_ERR_WORKSPACE = 6,  /* workspace missing, too small or misaligned          */
  Q1_ERR_CUDA = 7,       /* a CUDA runtime call or launch failed                */
  Q1_ERR_TIMEOUT = 8,    /* a bounded device-side wait ran out                  */
  Q1_ERR_DEVICE = 9      /* current device is not a compute capability 10.x GPU */
} q1_status;

typedef enum { Q1_BF16 = 0, Q1_F16 = 1, Q1_F32 = 2 } q1_dtype;

/* Type of the scales and biases.  fp16 is the rMLX checkpoint's ("The good
 * news - packing is standard": scales+biases F16); bf16 is the Bonsai image
 * checkpoint's ("1-bit Bonsai Image support", MLX-Gen backlog, "Context": BF16
 * scales/biases, bits 1, group_size 128).  Both widen to fp32 exactly, and all
 * arithmetic on them is the same. */
typedef enum { Q1_META_F16 = 0, Q1_META_BF16 = 1 } q1_meta_dtype;

/* One packed Q1 weight.  All pointers are device pointers owned by the caller.
 *   w: 16-byte aligned.  scales/biases: 2-byte aligned, meta_dtype each.
 *   N >= 1, K >= 128, K % 128 == 0.
 *   group_size: 128 (every checkpoint on the pages), or 32 or 64 (MLX's affine
 *   format allows them; "1-bit affine weight support", rMLX issue #207, lists
 *   "group_size=32 occupancy" among mlx#3161's edge cases).  scales/biases are
 *   then [N][K/group_size].  Every call takes all three; the gate and up
 *   matrices of one FFN (q1_ffn_fused*, q1_decode_chain) must share a group
 *   size (else Q1_ERR_GROUP).  The narrow products (M <= 8) close their MMA
 *   chains on every group: 128 is their fast path, 64 and 32 cost more
 *   instructions per weight (each step then covers one 32-weight word).
 *   meta_dtype: Q1_META_F16 (0, so a zero-initialised field means fp16) or
 *   Q1_META_BF16; anything else returns Q1_ERR_DTYPE.
 * The prefill path (q1_qmm above the narrow threshold) builds fp16 weight
 * tiles: with bf16 metadata, dequantized values must lie within fp16's range
 * (|value| <= 65504), as every fp16 checkpoint's do. */
typedef struct {
  const uint32_t *w;
  const uint16_t *scales;
  const uint16_t *biases; /* NULL => symmetric metadata */
  int64_t N;
  int64_t K;
  int32_t group_size;
  int32_t meta_dtype;     /* q1_meta_dtype */
} q1_weight;

/* ---- pack / unpack (rMLX issue #207, "packing is standard") ------------- */
/* bits uint8 [N][K] (bit 0 of every byte is the weight; other bits ignored)
 * -> w uint32 [N][K/32], LSB first.  K % 32 == 0.  Both 16-byte aligned. */
q1_status q1_pack(const uint8_t *bits, int64_t N, int64_t K, uint32_t *w, q1_stream stream);
/* w uint32 [N][K/32] -> bits uint8 [N][K] of 0/1 values.  Both 16-byte aligned. */
q1_status q1_unpack(const uint32_t *w, int64_t N, int64_t K, uint8_t *bits, q1_stream stream);

/* ---- dequantize (higgs PR #212, "What"; rMLX issue #207, the missing
 * affine_dequantize kernel) ---------------------------------------------- */
/* out [N][K] in out_t (bf16 / f16 / f32): the fp32 dequantized value rounded
 * once to nearest-even.  out 16-byte aligned.  Bit-exact. */
q1_status q1_dequantize(const q1_weight *W, q1_dtype out_t, void *out, q1_stream stream);

/* ---- exact repack from dense ("Bonsai masked gemv", cactus PR #775: tensors
 * whose 128-groups hold exactly {-s,+s} are repacked with the checkpoint's own
 * scales and zero quantization error; non-binary tensors are not) -----------
 * dense [N][K] in in_t (Q1_BF16, Q1_F16 or Q1_F32), device, 16-byte aligned.
 * Writes w [N][K/32] (16-byte aligned), scales [N][K/128] fp16 and, unless
 * biases is NULL, biases [N][K/128] fp16.  biases == NULL asks for the
 * symmetric form.  Per group of 128, values are compared by bit pattern (+0
 * and -0 differ; a NaN or infinity refuses the group):
 *   - more than two values: refused;
 *   - two values lo < hi (-0 < +0): bit 1 where the value is hi;
 *       symmetric: scale = RN16(-2 lo), kept if -0.5*scale == lo and
 *         fl32(scale - 0.5*scale) == hi bit for bit;
 *       affine: bias = RN16(lo), which must equal lo; scale = the first of
 *         RN16(fl32(hi - lo)), one fp16 step down, one up, two down, two up
 *         with fl32(scale + bias) == hi bit for bit;
 *   - one value v: symmetric: scale = RN16(2v) with all bits 1 when v's sign
 *     bit is clear, else RN16(-2v) with all bits 0 (kept if exact); affine:
 *     bias = v (must be an fp16 value), scale = +0, all bits 0.
 * A kept group dequantizes (q1_dequantize with out_t = in_t) to exactly the
 * input bits.  A refused group gets zero words, scale and bias and adds 1 to
 * *d_bad_groups (device int32, required; the caller zeroes it). */
q1_status q1_pack_from_dense(const void *dense, q1_dtype in_t, int64_t N, int64_t K, uint32_t *w,
                             uint16_t *scales, uint16_t *biases, int32_t *d_bad_groups,
                             q1_stream stream);

/* ---- matmul: y[M][N] = x[M][K] . Wd^T ------------------------------------
 * fp32 accumulation; x and y in `dtype` (bf16, fp16 or fp32, see above).
 * x and y 16-byte aligned.
 * q1_qmv: the M = 1 decode product (higgs PR #212, "What": the Q1 decode tile).
 * q1_qmm_narrow: 1 <= M <= 8 (speculative-verifier windows) with the weights
 *   kept packed and no dense temporary (higgs PR #212, "What": narrow Q1
 *   matrix multiplies of up to 8 flattened rows).  Leading dimensions are
 *   flattened by the caller: x [B][T][K] is passed as M = B*T.
 * q1_qmm: any M >= 1.  M <= q1_get_qmm_max_rows() runs the narrow path.
 *   At the default threshold (8), 9 <= M <= 16 also runs it, as two
 *   launches of 8 and M - 8 rows (no workspace needed): at these sizes that
 *   is faster than the prefill path.  Wider M runs the prefill path, which dequantizes weight stages straight
 *   into tensor memory and multiplies them on the tcgen05 tensor cores of CTA
 *   pairs (no dense weight temporary).  Its operands are fp16: symmetric
 *   weights are exact and affine ones rounded once at 2^-11; the activations
 *   enter as fp16 rows scaled by a power of two per row (kept in the
 *   workspace), which is exact for every activation whose scaled value is a
 *   normal fp16 number.
 * The narrow kernel covers K <= 40960 (a cluster of at most 8 CTAs, each
 * holding at most 10 spans of 512 k): q1_qmv and q1_qmm_narrow return
 * Q1_ERR_SHAPE above it, and q1_qmm runs such K on the prefill path for any
 * M (workspace required). */
q1_status q1_qmv(const q1_weight *W, const void *x, q1_dtype dtype, void *y, q1_stream stream);
q1_status q1_qmm_narrow(const q1_weight *W, const void *x, int64_t M, q1_dtype dtype,
                        void *y, q1_stream stream);
/* Workspace of q1_qmm: fp16 activation rows and per-row scales of the prefill
 * path (M*K*2 + M*4 bytes, each part rounded up to 256), plus, when the
 * prefill plan for this shape and device shares tiles between CTA pairs,
 * their fp32 partial sums (two tiles of 256 rows per pair) and a count per
 * tile.  The size depends on the current device and on q1_set_prefill_plan:
 * take it after both are set.  The call needs the workspace only on the
 * prefill path (M > q1_get_qmm_max_rows(), except 9..16 rows at the default
 * threshold, or K > 40960); workspace may be NULL otherwise. */
size_t q1_qmm_workspace_size(int64_t M, int64_t N, int64_t K);
q1_status q1_qmm(const q1_weight *W, const void *x, int64_t M, q1_dtype dtype, void *y,
                 void *workspace, size_t workspace_bytes, q1_stream stream);
/* Narrow/wide threshold (higgs PR #212, "Limitations": HIGGS_BONSAI_QMM_MAX_ROWS,
 * default 8).  Values are clamped to [0, 8].  The environment variable
 * Q1_QMM_MAX_ROWS, if set, gives the initial value when the library loads. */
void q1_set_qmm_max_rows(int rows);
int q1_get_qmm_max_rows(void);
/* Tiling of the prefill path (no counterpart on the pages; a tuning and test
 * control).  By default (0, 0) each call picks it from the shape: tiles of
 * 256 weight rows x token_tile tokens, token_tile a multiple of 16 in
 * [16, 256], and a schedule: split = 1 gives each CTA pair whole tiles in
 * turn; split = 2..4 shares each tile among that many pairs of a cluster,
 * which take contiguous k ranges and sum their partial tiles in a fixed
 * order; split = 0 gives each pair an equal run of (tile, k range) work, a
 * tile shared by neighbouring runs being summed in k order through the
 * workspace.  A pair set here is used by every later prefill call (with
 * split > 1, by those whose K holds at least 2 * split groups of 128, and
 * with split = 0, by those with fewer than 2^31 (tile, 128-k step) units;
 * others fall back to the automatic choice); values outside those ranges
 * restore the automatic choice.  Results are the same for every tiling up to the fp32
 * summation order. */
void q1_set_prefill_plan(int token_tile, int split);

/* ---- embedding gather (higgs PR #212, "What": Q1 embeddings) --------------
 * out[t][:] = dequant(E row ids[t]) in out_t, bit-exact like q1_dequantize.
 * ids: device int32 [T].  An id outside [0, E->N) gives a zero row and, when
 * d_bad_count is not NULL, adds 1 to *d_bad_count (device int32).  T >= 0
 * (T == 0 launches nothing).  out 16-byte aligned. */
q1_status q1_embed_gather(const q1_weight *E, const int32_t *ids, int64_t T, q1_dtype out_t,
                          void *out, int32_t *d_bad_count, q1_stream stream);

/* ---- fused dense FFN (higgs PR #212, "What": fused dense-FFN operations) ---
 * y[M][D] = Down . (SiLU(Gate . x) * (Up . x)) with SiLU(g) = g / (1 + e^-g).
 * gate, up: [F][D]; down: [D][F].  1 <= M <= 8; D, F <= 40960.  x [M][D], y [M][D]
 * in `dtype` (bf16, fp16 or fp32).
 * The intermediate h [M][F] is kept in bf16 at the start of the workspace
 * (q1_ffn_workspace_size(M, D, F) bytes, 256-byte aligned); it is still
 * there when the call's work completes. */
size_t q1_ffn_workspace_size(int64_t M, int64_t D, int64_t F);
q1_status q1_ffn_fused(const q1_weight *gate, const q1_weight *up, const q1_weight *down,
                       const void *x, int64_t M, q1_dtype dtype, void *y, void *workspace,
                       size_t workspace_bytes, q1_stream stream);

/* ---- fused FFN without any allocation ---------------------------------------
 * The source method has no counterpart of this call: it exists for callers
 * that must not allocate memory at all, not even a workspace.  It computes
 * exactly what q1_ffn_fused computes (same kernels, same results) and keeps h
 * in a fixed array inside this library instead of a caller workspace:
 *   - the array holds Q1_FFN_NOALLOC_BYTES (512 KiB) per device, so the call
 *     needs M * F * 2 <= Q1_FFN_NOALLOC_BYTES (e.g. M <= 8 with F <= 32768);
 *     larger shapes return Q1_ERR_WORKSPACE and launch nothing;
 *   - the call allocates nothing (no cudaMalloc / cudaFree, no allocating
 *     library call);
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and caches it: make that first call before any
 *     stream capture on that device;
 *   - nothing in the array has to start at zero: the gate/up kernel writes
 *     all of h before the down kernel reads it;
 *   - the array is shared by every call on the device: calls that can
 *     overlap in time (other streams, other host threads) race on it, so
 *     order them (one stream, or events);
 *   - h of the last call stays in the array until the next call. */
#define Q1_FFN_NOALLOC_BYTES (512u * 1024u)
q1_status q1_ffn_fused_noalloc(const q1_weight *gate, const q1_weight *up, const q1_weight *down,
                               const void *x, int64_t M, q1_dtype dtype, void *y, q1_stream stream);

/* ---- synthetic decode chain -----------------------------------------------
 * The Q1 linears of a decode step, layer after layer ("Support Bonsai-27B
 * affine Q1", higgs PR #212, section "Measured impact": decode time of a
 * model whose linears are all Q1; no attention, norms or residuals, so it is
 * not a model).  For l = 0 .. n_layers-1, with h_0 = x:
 *   a       = attn_l . h_l                               (the narrow product)
 *   h_{l+1} = down_l . (SiLU(gate_l . a) * (up_l . a))   (the fused FFN)
 * and y = h_{n_layers}.  Every intermediate is bf16, and the result is exactly
 * that of the same q1_qmm_narrow and q1_ffn_fused calls made one by one (same
 * kernels, same order).  All launches are chained with programmatic dependent
 * launch, so each one streams its weights while its predecessor drains.
 * layers: host array of n_layers >= 1 entries (the weights inside are device
 * memory).  Every layer has the same D (attn [D][D]; gate, up [F_l][D];
 * down [D][F_l]); F_l may differ.  1 <= M <= 8; D, F_l <= 40960.
 * x, y [M][D] bf16, 16-byte aligned; y must not overlap x or the workspace.
 * Workspace: q1_decode_chain_workspace_size(M, D, max F_l) bytes, 256-byte
 * aligned (a, the current h and the FFN intermediate). */
typedef struct {
  q1_weight attn; /* [D][D] */
  q1_weight gate; /* [F][D] */
  q1_weight up;   /* [F][D] */
  q1_weight down; /* [D][F] */
} q1_decode_layer;
size_t q1_decode_chain_workspace_size(int64_t M, int64_t D, int64_t F_max);
q1_status q1_decode_chain(const q1_decode_layer *layers, int32_t n_layers, const void *x,
                          int64_t M, q1_dtype dtype, void *y, void *workspace,
                          size_t workspace_bytes, q1_stream stream);

/* ---- symmetric check (higgs PR #212, walkthrough: symmetric bias
 * compaction and validation) -------------------------------------------------
 * Writes 1 to *d_is_symmetric (device int32) iff every stored bias equals
 * -scale/2 exactly in fp32 (+0 == -0; NaN never equal), else 0.
 * W->biases must not be NULL. */
q1_status q1_check_symmetric(const q1_weight *W, int32_t *d_is_symmetric, q1_stream stream);

/* ---- diagnostics ------------------------------------------------------------ */
/* Synchronizes `stream`, then reads and clears the device error words of the
 * library's kernels.  *flags (may be NULL) receives their OR; returns
 * Q1_ERR_TIMEOUT if any bounded wait ran out since the last call. */
q1_status q1_device_errors(unsigned int *flags, q1_stream stream);
const char *q1_status_string(q1_status s);
/* Controls of the bounded waits (no counterpart on the pages; for tests of
 * the timeout path).  Every wait of the narrow and prefill kernels on another
 * role's progress is bounded; one that runs out sets the device error word
 * (bit 0: prefill kernels, bit 1: narrow kernels).  Later waits of the
 * prefill kernels then give up at once until q1_device_errors reads the word;
 * those of the narrow kernels each run out on their own limit.
 * q1_set_wait_limit_ns: the bound, in ns of the GPU's global timer (default
 *   2 s; 0 restores it).
 * q1_set_stalled_producers: nonzero makes the producers of later launches
 *   issue no copies, so that every wait for their data runs out; no copy is
 *   then in flight when the kernels give up.  The results of such launches
 *   are undefined; 0 restores normal launches.
 * Both apply to the current device, to launches made after the call, and
 * synchronize with the device; they are not meant to race with launches on
 * other threads. */
q1_status q1_set_wait_limit_ns(uint64_t ns);
q1_status q1_set_stalled_producers(int stall);

#ifdef __cplusplus
}
#endif
#endif /* Q1_H_ */
