/*
 * sl.h -- C ABI of libsl, the B300 (sm_103a) layer-streamed NF4 LoRA library.
 *
 * What it computes (sources by page title and section):
 *  - LoRA fine-tuning on a frozen base held in NF4: "Exact Layer Streaming:
 *    LoRA Fine-Tuning of an 8B Model on a 4 GB Laptop GPU" (abstract);
 *    "Soup CLI Lets You Fine-Tune an 8B LLM on a 4 GB Laptop GPU" ("Key
 *    Takeaways": Llama-3.1-8B-Instruct + NF4).
 *  - Layer streaming: the frozen base stays in (pinned) host RAM and decoder
 *    layers are brought to the GPU for the forward and again, in reverse, for
 *    the backward ("Soup CLI ...", "How Layer Streaming Works"), through two
 *    device buffers ("Soup: Fine-Tuning an 8B LLM on a 4 GB Laptop GPU with One
 *    YAML File", "Layer Streaming: The Mechanism Behind the 4 GB Claim": a
 *    pinned base store and two VRAM buffers).  The streamed run must be
 *    bit-exact against a resident run of the same numerics ("Exact Layer
 *    Streaming ...", abstract; "Soup CLI ...", "v0.73.0: Fixing Silent Wrong
 *    Gradients").
 *  - The base is never upcast: it is consumed in its storage dtype ("Soup:
 *    Fine-Tuning ...", "The FP32 Bug and What It Means for Your VRAM"), and
 *    adapter gradients are fp32 ("Known Limitations and Failure Modes").
 *  - The cross-entropy over the LM head without the full logits ("Exact Layer
 *    Streaming ...", abstract: the logits term's bytes per element).
 *
 * Conventions for every call:
 *  - Device pointers unless stated; the CALLER owns every tensor passed in.
 *    libsl owns only what sl_stack_create allocates (two device layer buffers,
 *    a copy stream, a high-priority main stream, events), one high-priority
 *    stream per device (created on the first LoRA backward there) with a few
 *    events per thread, and two file-scope device arrays that every device
 *    loading the library holds until exit: the error word (two ints) and the
 *    4 MiB scratch of sl_lora_linear_fwd_noalloc.
 *  - Work is enqueued on the caller's stream and the call returns without
 *    waiting, except where a call says it synchronises.
 *  - bf16 tensors are passed as void* (IEEE bfloat16 bit patterns, row-major,
 *    densely packed); sizes are element counts.
 *  - Every call returns sl_status; on failure nothing is enqueued (argument
 *    errors) or the CUDA error is reported (SL_ERR_CUDA), and
 *    sl_last_error() (thread-local) describes it.  No C++ exception crosses
 *    the ABI.
 *  - Kernels never trap.  A bounded wait that gives up (after about two
 *    seconds) writes SL_ERR_TIMEOUT into the device error word and returns;
 *    sl_check_device_errors() reports it.
 */
#ifndef SL_H_
#define SL_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SL_OK = 0,
  SL_ERR_INVALID = 1,      /* bad argument: null pointer, shape, alignment, workspace too small */
  SL_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed */
  SL_ERR_UNSUPPORTED = 3,  /* valid but not implemented (e.g. no sm_103a device) */
  SL_ERR_TIMEOUT = 4,      /* a device-side bounded wait gave up */
  SL_ERR_NONFINITE = 5,    /* non-finite input where the operation forbids it */
  SL_ERR_OOM = 6           /* a libsl-owned allocation failed */
} sl_status;

typedef enum { SL_DTYPE_BF16 = 0, SL_DTYPE_F32 = 1 } sl_dtype;
typedef enum { SL_WEIGHT_NF4 = 0, SL_WEIGHT_BF16 = 1, SL_WEIGHT_NF4_DQ = 2 } sl_weight_kind;
typedef enum { SL_MODE_STREAMED = 0, SL_MODE_RESIDENT = 1 } sl_stack_mode;

/* A frozen base weight W [N, K] (N = out features, K = in features), the
 * layout of a PyTorch Linear.weight.
 *  kind = SL_WEIGHT_NF4:  codes  [N*K/2] bytes, row-major, element 2i in the
 *                         HIGH nibble of byte i; absmax [N*K/64] fp32, one per
 *                         64 consecutive elements of a row.  Needs K % 256 == 0.
 *  kind = SL_WEIGHT_BF16: w [N, K] bf16.
 *  kind = SL_WEIGHT_NF4_DQ: codes as for NF4; the absmax double-quantised
 *                         (sl_nf4_double_quantize): qabsmax int8 transposed,
 *                         element [j, dq_col0 + n] for row n and 64-block j,
 *                         rows of qabsmax_ld bytes; absmax2 fp32 (offset,
 *                         scale) pairs, pair [j, (dq_col0 + n) / 256] at
 *                         absmax2 + j * absmax2_ld + 2 * ((dq_col0 + n) / 256).
 *                         dq_col0 lets a weight be a column range of arrays
 *                         that several projections share.  Needs K % 256 == 0,
 *                         N and dq_col0 multiples of 256, and M > 128 in the
 *                         linear and group calls (the CTA-pair GEMM).
 * All pointers 16-byte aligned; N % 32 == 0; qabsmax_ld a multiple of 16,
 * absmax2_ld of 4. */
typedef struct {
  int32_t kind;
  int64_t N;
  int64_t K;
  const uint8_t* codes;
  const float* absmax;
  const void* w;
  const int8_t* qabsmax;  /* SL_WEIGHT_NF4_DQ only (NULL otherwise) */
  int64_t qabsmax_ld;
  const float* absmax2;
  int64_t absmax2_ld;
  int64_t dq_col0;
} sl_weight;

/* ---------------------------------------------------------------- library */

/* Thread-local description of the last failure in this thread ("" if none). */
const char* sl_last_error(void);

/* ABI version (major*10000 + minor*100 + patch). */
int32_t sl_version(void);

/* Kernels libsl has launched in this process so far (all devices and
 * threads); the difference over a region counts the region's launches. */
uint64_t sl_launch_count(void);

/* Host copy of the library's NF4 levels (16 fp32, ascending).  The levels are
 * the published NormalFloat-4 construction (QLoRA); the pages name NF4 but do
 * not print them.  Never fails. */
void sl_nf4_code_table(float out[16]);

/* Synchronises `stream`, then reads and clears this device's error word.
 * Returns SL_OK, or the code a kernel recorded (SL_ERR_TIMEOUT, ...). */
sl_status sl_check_device_errors(cudaStream_t stream);

/* Launches one kernel that waits on a device flag nothing ever sets, with a
 * wait limit of `limit_ns` nanoseconds (clamped to [1e3, 2e9]); the kernel
 * gives up, records SL_ERR_TIMEOUT in the error word and exits normally.
 * Exists so that tests can prove a bounded wait ends without faulting the
 * GPU.  `mbarrier` != 0 makes the wait an mbarrier wait instead of a flag
 * poll. */
sl_status sl_debug_timeout_probe(int64_t limit_ns, int32_t mbarrier, cudaStream_t stream);

/* Kernel timing for measurement.  enable != 0 clears earlier records and
 * starts recording a CUDA event pair, on the launching stream, around every
 * tensor-core launch; enable == 0 stops recording.  Costs one event pair
 * per launch.  Variants: 0 NF4 forward, 1 NF4 dX, 2 bf16 forward, 3 bf16
 * dX, 4 CE logits chunk (exp epilogue), 5 CE dH accumulation, 6 rank-r
 * T = X A^T, 7 rank-r U = dY B, 8 rank-r dA / dB, 9 attention forward,
 * 10 attention backward (its three kernels together). */
sl_status sl_kernel_timing(int32_t enable);

/* Totals over the launches of one variant recorded since timing was
 * enabled: launch count, summed device time in ms (waits for the recorded
 * events) and algorithmic work: FLOPs for the GEMM variants 0-5 (2 M N K,
 * plus 2 M N r for the folded LoRA side product), bytes for the rank-r
 * passes 6-8 (the large operand once, the rank-r operands and the output),
 * FLOPs for attention (2 x 128 per product per visible causal (query, key)
 * pair: 2 products forward; 5 backward, S recomputed once). */
sl_status sl_kernel_timing_read(int32_t variant, uint64_t* launches, double* ms, double* work);

/* The GEMM variants (0-5) timed on the device clock: every timed GEMM launch
 * records its own span, from the first CTA past its dependency wait to the
 * last CTA whose output stores have completed (%globaltimer), into a slot
 * buffer libsl allocates on the first sl_kernel_timing(1) (which therefore
 * synchronises the device).  Returns the launches that recorded a span and
 * their summed span in ms.  Unlike an event pair around a launch, the span
 * is not lengthened by delayed event timestamps (a host-to-device copy in
 * flight delays them by ~16 us per pair on B300). */
sl_status sl_kernel_timing_read_clock(int32_t variant, uint64_t* launches, double* ms);

/* ------------------------------------------------------------- NF4 (K0/K1) */

/* NF4-quantise W [N, K] (dtype SL_DTYPE_BF16 or SL_DTYPE_F32) into codes
 * [N*K/2] and absmax [N*K/64] (layouts of sl_weight).  Per 64-element block:
 * absmax = max |w|; x = w / absmax (IEEE fp32 division); code = nearest NF4
 * level to x, ties to the lower level; absmax == 0 gives code 7 (the zero
 * level) everywhere.  Requires K % 64 == 0, pointers 16-byte aligned.
 * SYNCHRONISES `stream` to read the non-finite flag: returns
 * SL_ERR_NONFINITE if any input is NaN or infinite (outputs then undefined). */
sl_status sl_nf4_quantize(const void* W, int32_t dtype, int64_t N, int64_t K,
                          uint8_t* codes, float* absmax, cudaStream_t stream);

/* Double quantisation of the absmax (QLoRA's 8-bit absmax: the pages' 3.60 GB
 * store and 113 MB layer buffers for Llama-3.1-8B, "Soup: Fine-Tuning ...",
 * "Layer Streaming: The Mechanism Behind the 4 GB Claim"; the format is this
 * library's reading): absmax [N, K/64] fp32 as written by sl_nf4_quantize ->
 * qabsmax[j * qabsmax_ld + n] int8 and, per 256 consecutive n of block j,
 * (c, s) at absmax2[j * absmax2_ld + 2 * (n / 256)]:
 *   c = fp32(float64 sum of the 256 values, ascending n) / 256),
 *   d = fp32(a - c), s = fp32(max |d| / 127),
 *   q = s == 0 ? 0 : clamp(rint(fp32(d / s)), -127, 127)  (ties to even);
 * the absmax a GEMM then uses is fma(s, q, c) rounded once.  N % 256 == 0,
 * K % 64 == 0; the output pointers may be column offsets into wider arrays
 * (see sl_weight); 16-byte aligned input. */
sl_status sl_nf4_double_quantize(const float* absmax, int64_t N, int64_t K, int8_t* qabsmax, int64_t qabsmax_ld,
                                 float* absmax2, int64_t absmax2_ld, cudaStream_t stream);

/* w_hat = fp32(T[code] * absmax), written as bf16 (rounded to nearest even)
 * or fp32 per `out_dtype`, out [N, K].  Requires K % 64 == 0. */
sl_status sl_nf4_dequantize(const uint8_t* codes, const float* absmax, int64_t N, int64_t K,
                            int32_t out_dtype, void* out, cudaStream_t stream);

/* The same for any sl_weight of kind NF4 or NF4_DQ (w_hat with the absmax the
 * GEMMs use: fma(s, q, c) for NF4_DQ). */
sl_status sl_weight_dequantize(const sl_weight* w, int32_t out_dtype, void* out, cudaStream_t stream);

/* ------------------------------------------------------ LoRA linear (a3-a6) */

/* Forward of the frozen-base LoRA linear
 *     Y = X W^T + s (X A^T) B^T,    s = alpha / r,
 * X [M, K] bf16, A [r, K] bf16, B [N, r] bf16, Y [M, N] bf16 (fp32
 * accumulation, one rounding).  T_save [M, r] fp32 receives X A^T (kept for
 * the backward; the side product s T B^T is folded into the same
 * accumulator with fp32 accuracy); may be NULL only when r == 0; 16-byte
 * aligned (it is read by TMA).  r == 0 (or A == B == NULL) computes the base
 * alone -- the adapters-off pass.  r <= 32, r % 8 == 0.  `ws` may be NULL;
 * given a buffer of sl_lora_linear_workspace_size bytes (256-byte aligned),
 * the forward uses the part after U to split the GEMM's last partial wave
 * of tiles along K (pieces' fp32 partial sums added in a fixed order: the
 * result is bitwise reproducible, and equal to the unsplit one up to fp32
 * summation order). */
sl_status sl_lora_linear_fwd(const sl_weight* w, const void* X, int64_t M,
                             const void* A, const void* B, int32_t r, float alpha,
                             void* Y, void* T_save, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* Backward of the linear above for upstream gradient dY [M, N] bf16:
 *     U = dY B (fp32);  dX = dY W + s U A;  dA = s U^T X;  dB = s dY^T T_save,
 * T_save [M, r] fp32 from the forward.
 * dX [M, K] bf16 (may be NULL to skip); dA [r, K] and dB [N, r] fp32,
 * overwritten when accumulate == 0, added to otherwise.  Every reduction
 * runs in a fixed order: results are bitwise reproducible.  `ws` must hold
 * U [M, r] fp32 (256-byte aligned): it carries U between the rank-r passes;
 * with sl_lora_linear_workspace_size(M, N, K, r) bytes the rest serves the
 * dX GEMM's split-K scratch as in the forward.  U and the dX GEMM run on a
 * high-priority library stream and dA, dB on `stream` beside them; the call
 * leaves `stream` ordered after all of it. */
sl_status sl_lora_linear_bwd(const sl_weight* w, const void* X, const void* dY, int64_t M,
                             const void* A, const void* B, int32_t r, float alpha,
                             const void* T_save, void* dX, float* dA, float* dB,
                             int32_t accumulate, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* The forward above for callers that cannot allocate device memory -- code
 * running under a memory manager that owns all device memory (a framework's
 * caching allocator with a hard budget, or an embedding application that
 * forbids cudaMalloc because it synchronises the device and fragments its
 * pool) and therefore cannot pass a workspace.  No counterpart on the pages:
 * it exists for those callers only.  Same arguments and results as
 * sl_lora_linear_fwd without `ws`; the call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).  Its scratch, the K-split partial
 * sums of X A^T, lives in one fixed 4 MiB device array inside libsl that
 * every device loading the library holds until exit; a call needing more
 * than 4 MiB (ceil(K/512) * M * r * 4 bytes) returns SL_ERR_INVALID and
 * enqueues nothing, as does a base pointer (X, A, B, Y, T_save) that is not
 * 16-byte aligned.  The first call on a device looks up the device
 * addresses of that array and of the error word (cudaGetSymbolAddress) and
 * should come before any stream capture.  All calls share the array and it keeps the last call's
 * contents (nothing in it needs to start at zero); calls that overlap on
 * the GPU, e.g. on two streams, race on it and must be serialised. */
sl_status sl_lora_linear_fwd_noalloc(const sl_weight* w, const void* X, int64_t M,
                                     const void* A, const void* B, int32_t r, float alpha,
                                     void* Y, void* T_save, cudaStream_t stream);

/* Workspace bytes of one linear call: the backward's U [M, r] fp32, rounded
 * up to 256, then, when M > 128, the CTA-pair GEMM's split-K scratch (a
 * fixed ~19 MB on a 148-SM B300: a flag and a 256 KB fp32 partial tile per
 * SM pair); 0 when r == 0. */
size_t sl_lora_linear_workspace_size(int64_t M, int64_t N, int64_t K, int32_t r);

/* ------------------------------------------------------ projection groups */

/* The forward of G (<= 4) LoRA linears that read the same input X -- in a
 * decoder layer ("Soup CLI ...", "How Layer Streaming Works") the q, k, v
 * projections or gate, up -- as one fused GEMM plus one rank-r pass:
 *     Y_g = X W_g^T + s (X A_g^T) B_g^T,  s = alpha / r,  g = 0 .. G-1.
 * The pages describe no such grouping; it is how this library runs a
 * layer's projections that share an input, with the same arithmetic as G
 * calls of sl_lora_linear_fwd up to fp32 summation order.  Layout: w_cat is
 * one NF4 weight of N = sum N_g rows (the projections' weights back to back,
 * N_g multiples of 256); A_cat [G r, K] and B_cat [sum N_g, r] bf16 are the
 * adapters back to back; Y_cat [M, sum N_g] bf16 holds Y_g in columns
 * [N_0 + .. + N_{g-1}, + N_g); T_cat [M, G r] fp32 (16-byte aligned) holds
 * X A_g^T in columns [g r, g r + r).  Requires NF4, 128 < M, r % 8 == 0,
 * r <= 32, G r <= 64 (SL_ERR_INVALID otherwise); r == 0 runs the bases
 * alone (adapters off; A_cat, B_cat, T_cat may be NULL).  Allocates nothing. */
sl_status sl_lora_group_fwd(const sl_weight* w_cat, int32_t G, const int64_t* N_g,
                            const void* X, int64_t M, const void* A_cat, const void* B_cat,
                            int32_t r, float alpha, void* Y_cat, void* T_cat, cudaStream_t stream);

/* The backward of the group above for dY_cat [M, sum N_g] bf16 (dY_g in the
 * columns of Y_g):  dX = sum_g (dY_g W_g + s U_g A_g) with U_g = dY_g B_g
 * (one fused GEMM), dA_cat [G r, K] (rows of adapter g = s U_g^T X) and
 * dB_cat [sum N_g, r] (rows of projection g = s dY_g^T T_g), fp32,
 * overwritten when accumulate == 0, added to otherwise.  dX [M, K] bf16 may
 * be NULL.  `ws` must hold U_cat [M, G r] fp32 (256-byte aligned); with
 * sl_lora_group_workspace_size(M, G, r) bytes the rest serves the dX GEMM's
 * split-K scratch (as in sl_lora_linear_fwd).  r == 0: dX of the bases
 * only.  Reductions run in a fixed order: results are bitwise
 * reproducible.  Streams as in sl_lora_linear_bwd. */
sl_status sl_lora_group_bwd(const sl_weight* w_cat, int32_t G, const int64_t* N_g,
                            const void* X, const void* dY_cat, int64_t M,
                            const void* A_cat, const void* B_cat, int32_t r, float alpha,
                            const void* T_cat, void* dX, float* dA_cat, float* dB_cat,
                            int32_t accumulate, void* ws, size_t ws_bytes, cudaStream_t stream);

size_t sl_lora_group_workspace_size(int64_t M, int32_t G, int32_t r);

/* ------------------------------------------------- streamed stack (a2-a7) */

/* Byte layout of one layer blob (the unit that is streamed): the seven
 * projections q, k, v, o, gate, up, down of a decoder layer with hidden D,
 * kv width Dkv and MLP width F.  NF4: the seven projections' codes in that
 * order, then their absmax in that order; BF16: the seven weights in order.
 * With the size rules below every region is a multiple of 256 bytes, so the
 * q, k, v and the gate, up weights each lie back to back (one weight of
 * N = D + 2 Dkv or 2 F rows, as the projection groups use them).
 * offsets[2p] / offsets[2p+1] receive the byte offsets of projection p's
 * codes / absmax (NF4) or of its weight / 0 (BF16), every offset 256-byte
 * aligned; *blob_bytes the total.
 * NF4_DQ (the 8-bit absmax that makes the pages' 113 MB layer buffer and
 * 3.60 GB base store for Llama-3.1-8B: "Soup: Fine-Tuning ...", "Layer
 * Streaming: The Mechanism ..."): the codes as for NF4, then for each of the
 * four absmax groups q/k/v, o, gate/up, down (projections that read one
 * input) its qabsmax int8 [K/64, N_group] and its absmax2 fp32
 * [K/64, round_up(2 N_group / 256, 4)] (sl_nf4_double_quantize of the
 * group's fp32 absmax, rows of its projections in order); offsets[2p+1] is
 * the qabsmax array of projection p's group.  Needs Dkv % 256 == 0.
 * Every kind ends with the layer's two RMS-norm weights, fp32 [D] each:
 * offsets[14] (before the attention / mixing step) and offsets[15] (before
 * the MLP); all ones reproduce the unweighted norm exactly. */
sl_status sl_stack_blob_layout(int32_t kind, int64_t D, int64_t Dkv, int64_t F,
                               size_t offsets[16], size_t* blob_bytes);

/* The double-quantised absmax of an NF4_DQ layer blob, per projection p:
 * its group's qabsmax at byte q_off[p] (rows of q_ld[p] bytes), absmax2 at
 * byte a2_off[p] (rows of a2_ld[p] floats), and the projection's first
 * column col0[p] in both (its sl_weight's dq_col0).  Same size rules as
 * sl_stack_blob_layout for NF4_DQ. */
sl_status sl_stack_dq_layout(int64_t D, int64_t Dkv, int64_t F, size_t q_off[7], int64_t q_ld[7],
                             size_t a2_off[7], int64_t a2_ld[7], int64_t col0[7]);

typedef enum { SL_MIX_TOKEN_LOCAL = 0, SL_MIX_ATTENTION = 1 } sl_mixer;

typedef struct {
  int32_t L;                        /* number of layers */
  int32_t kind;                     /* SL_WEIGHT_NF4, SL_WEIGHT_NF4_DQ (M > 128 only) or SL_WEIGHT_BF16 */
  int64_t D, Dkv, F;                /* hidden, kv width (multiple of 128), MLP width */
  const void* const* host_blobs;    /* L pointers to PINNED host blobs (sl_stack_blob_layout) */
  const void* const* device_blobs;  /* L device copies for SL_MODE_RESIDENT, or NULL */
  int32_t mixer;                    /* SL_MIX_TOKEN_LOCAL (0) or SL_MIX_ATTENTION */
  int64_t seq_len;                  /* attention: tokens per sequence (multiple of 128; M % seq_len == 0) */
  double rope_theta;                /* attention: rotary base (500000 for Llama-3.1) */
} sl_stack_desc;

typedef struct sl_stack sl_stack;

/* Creates a stack handle: checks that every host blob is page-locked
 * (cudaPointerGetAttributes; pageable memory -> SL_ERR_INVALID), allocates
 * the two device layer buffers, a copy stream, a main stream at the highest
 * priority and the events on the current device.  The pre-flight report ("Soup: Fine-Tuning ...", "Layer
 * Streaming: The Mechanism ...") comes back in *host_bytes (L * blob bytes)
 * and *buffer_bytes (the two buffers together).  The descriptor's pointer
 * arrays are copied; the blobs themselves stay owned by the caller and must
 * outlive the handle. */
sl_status sl_stack_create(const sl_stack_desc* desc, sl_stack** out,
                          size_t* host_bytes, size_t* buffer_bytes);
sl_status sl_stack_destroy(sl_stack* s);

/* Workspace for sl_stream_stack_step at M tokens and rank r. */
size_t sl_stack_workspace_size(const sl_stack* s, int64_t M, int32_t r);

/* One training step of the stack:
 *  forward layers 0..L-1 from h0 [M, D] fp32 to hL [M, D] fp32, then
 *  backward L-1..0 from dh_top [M, D] fp32 to dh0 [M, D] fp32, writing for
 *  every layer l and projection p (index 7*l + p, order q k v o gate up down)
 *  dA[7l+p] [r, K_p] fp32 and dB[7l+p] [N_p, r] fp32 (overwritten when
 *  accumulate == 0, added to otherwise: gradient accumulation over
 *  micro-batches, each of which re-streams the base -- "Exact Layer
 *  Streaming ..." (abstract): accumulation is per-token I/O-neutral).
 *  A[7l+p] [r, K_p] bf16 and B[7l+p] [N_p, r] bf16 are the adapters; r == 0
 *  (A, B, dA, dB may then be NULL) runs the frozen base alone, the
 *  adapters-off reference pass ("Soup CLI ...", "Key Takeaways": preference
 *  training with the streamed base and adapters off).
 * The layer is a pre-norm decoder layer: weighted RMS norm (weights in the
 * blob), q/k/v, the mixing step, o, weighted RMS norm, SiLU-gated MLP, fp32
 * residual stream, bf16 GEMM inputs/outputs.  Mixing: SL_MIX_ATTENTION is
 * causal grouped-query attention with rotary positions (sl_attention_fwd:
 * q and k rotated in place, the saved q/k are the rotated ones);
 * SL_MIX_TOKEN_LOCAL is a = q*rep(k) + rep(v).
 * SL_MODE_STREAMED: layer l is copied from its pinned host blob into device
 * buffer l % 2 on the handle's copy stream; CUDA events order each copy
 * after the last kernel that read the buffer and each layer's kernels after
 * its copy.  The backward reuses the two layers already resident at the
 * turn.  SL_MODE_RESIDENT: the same kernels, in the same order, read the
 * descriptor's device_blobs; results are bitwise identical.  The step runs
 * on the handle's main stream once `stream` reaches the call; every
 * projection's dA and dB passes run on `stream` beside the next kernels,
 * and `stream` is ordered after the whole step when the call returns.
 * `ws` must hold sl_stack_workspace_size(s, M, r) bytes, 256-byte aligned. */
sl_status sl_stream_stack_step(sl_stack* s, int32_t mode, const float* h0, int64_t M,
                               const float* dh_top, const void* const* A,
                               const void* const* B, int32_t r, float alpha,
                               float* hL, float* dh0, float* const* dA, float* const* dB,
                               int32_t accumulate, void* ws, size_t ws_bytes, cudaStream_t stream);

/* One complete supervised fine-tuning step on top of the stack:
 * h0 = embed[tokens] (embed [V, D] bf16, tokens [M] int32; a token outside
 * [0, V) gives a zero row and SL_ERR_INVALID in the device error word), the
 * stack forward, x = bf16(RMS(hL) * norm_final) (norm_final fp32 [D] or
 * NULL), the mean cross-entropy of x against W_head [V, D] bf16 with
 * labels [M] int32 (-100 ignored; sl_ce_fwd_bwd, vocab chunks of chunk_V)
 * into *loss (one fp32 on the device), its gradient back through the final
 * norm, and the stack backward into dA, dB as sl_stream_stack_step.  The
 * embedding and the head stay on the device; the layers stream as in
 * sl_stream_stack_step.  `ws`: sl_sft_workspace_size bytes, 256-byte
 * aligned. */
sl_status sl_sft_step(sl_stack* s, int32_t mode, const int32_t* tokens, const int32_t* labels, int64_t M,
                      const void* embed, int64_t V, const float* norm_final, const void* W_head, int64_t chunk_V,
                      const void* const* A, const void* const* B, int32_t r, float alpha, float* loss,
                      float* const* dA, float* const* dB, int32_t accumulate, void* ws, size_t ws_bytes,
                      cudaStream_t stream);
size_t sl_sft_workspace_size(const sl_stack* s, int64_t M, int32_t r, int64_t V, int64_t chunk_V);

/* Host-side counters of the last step on this handle: bytes copied host to
 * device and the number of libsl kernels launched. */
sl_status sl_stack_last_step_stats(const sl_stack* s, uint64_t* h2d_bytes, uint64_t* kernels);

/* ------------------------------------- attention of the full decoder layer */
/* Causal grouped-query attention with rotary positions, the token mixing of
 * a Llama-shaped decoder layer (the pages name Llama-3.1-8B and Qwen2.5-3B
 * but do not describe the layer: "Soup CLI Lets You Fine-Tune an 8B LLM
 * ...", "How Layer Streaming Works").  Layout: M rows = M / S sequences of S
 * tokens (S % 128 == 0), positions 0..S-1 in every sequence; q [M, H*128],
 * k and v [M, Hkv*128] bf16 with row strides (elements, multiples of 8,
 * 16-byte aligned bases); query head h reads kv head h / (H / Hkv); scores
 * q . k / sqrt(128), causal inside each sequence. */

/* Rotary table for positions 0..S-1: table[p*128 + i] = cos(p theta^(-i/64)),
 * table[p*128 + 64 + i] = sin(p theta^(-i/64)), i < 64; fp32 [S, 128],
 * computed in fp64. */
sl_status sl_rope_table(int64_t S, double theta, float* table, cudaStream_t stream);

/* In place on x [M, nheads*128] bf16 (row stride ld): the pairs (i, i + 64)
 * of every head rotated by the angle of the row's position (row % S), or by
 * its negative (inverse != 0), in fp32, rounded once to bf16. */
sl_status sl_rope_apply(void* x, int64_t ld, int64_t M, int32_t nheads, int64_t S, const float* table,
                        int32_t inverse, cudaStream_t stream);

/* o [M, H*128] bf16 (row stride ldo) = softmax(q k^T / sqrt(128) + causal
 * mask) v per head, and lse [H, M] fp32 (head-major) = the natural log of
 * each row's softmax normaliser.  One kernel (tcgen05: S and P V on the
 * tensor cores, the online softmax in registers). */
sl_status sl_attention_fwd(const void* q, int64_t ldq, const void* k, int64_t ldk, const void* v, int64_t ldv,
                           int64_t M, int64_t S, int32_t H, int32_t Hkv, void* o, int64_t ldo, float* lse,
                           cudaStream_t stream);

/* Bytes of the backward's workspace: Di [H, M] fp32 and the per-query-head
 * fp32 partials of dK and dV [H, M, 128] each. */
size_t sl_attention_workspace_size(int64_t M, int32_t H);

/* The backward given o, lse of the forward and dO = dL/do (bf16, row
 * stride lddo): dq [M, H*128], dk and dv [M, Hkv*128] bf16, each written
 * once (dk, dv: per-query-head partials summed over the query heads of
 * their kv head in head order: bitwise reproducible).  rope_table (nullable, sl_rope_table): dq and dk
 * leave rotated by the inverse angle, i.e. they are the gradients of q and
 * k before sl_rope_apply.  ws: sl_attention_workspace_size bytes, 16-byte
 * aligned. */
sl_status sl_attention_bwd(const void* q, int64_t ldq, const void* k, int64_t ldk, const void* v, int64_t ldv,
                           const void* o, int64_t ldo, const void* dO, int64_t lddo, const float* lse, int64_t M,
                           int64_t S, int32_t H, int32_t Hkv, void* dq, int64_t lddq, void* dk, int64_t lddk,
                           void* dv, int64_t lddv, const float* rope_table, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* ------------------------------------------------ LM-head cross-entropy (a8) */

/* loss = (1/N_valid) sum over rows with labels[i] != ignore_index of
 * (logsumexp_v z_iv - z_i,label), z = H W_head^T;
 * dH = (softmax(z) - onehot(label)) W_head / N_valid on valid rows, 0 elsewhere.
 * H [M, D] bf16, W_head [V, D] bf16, labels [M] int32 (in [0, V) or
 * ignore_index), loss: ONE fp32 on the device, dH [M, D] fp32 (the residual
 * stream's gradient dtype; it can feed sl_stream_stack_step's dh_top).  The
 * vocab is processed in chunks of chunk_V (multiple of 256) rows of W_head;
 * no [M, V] logits tensor ever exists, only an [M, chunk_V] bf16 softmax
 * chunk and O(M * V / 256) per-tile partials in `ws` (plus, for M > 128, a
 * fixed ~19 MB scratch in which the CTA-pair GEMMs split their last partial
 * wave along K).  N_valid == 0 gives
 * loss 0 and dH 0.  D % 256 == 0, V % 32 == 0.  A label outside [0, V) that
 * is not ignore_index is treated as ignored and recorded as SL_ERR_INVALID
 * in the device error word.  `ws` must hold sl_ce_workspace_size(M, D, V,
 * chunk_V) bytes, 256-byte aligned. */
sl_status sl_ce_fwd_bwd(const void* H, int64_t M, int64_t D, const void* W_head, int64_t V,
                        const int32_t* labels, int32_t ignore_index, int64_t chunk_V,
                        float* loss, float* dH, void* ws, size_t ws_bytes, cudaStream_t stream);

size_t sl_ce_workspace_size(int64_t M, int64_t D, int64_t V, int64_t chunk_V);

#ifdef __cplusplus
}
#endif
#endif /* SL_H_ */
