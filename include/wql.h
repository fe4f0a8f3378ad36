/*
 * wql.h -- C ABI of the weight-only quantised lm_head library (libwql.so).
 *
 * One operation and its load-time preparation:
 *
 *   logits[m, n] = sum_k x[m, k] * q[n, k] * s[n, k / G]   (+ bias[n])
 *
 * with Wq symmetric int4 (nibble = q + 8, q in [-8, 7]) or int8 (q in
 * [-127, 127]) and one fp16/bf16 scale per group of G hidden columns or per
 * row.  The dense weight is never materialised.  Sources:
 *   - "Fused WNA16 GEMM for tied quantized lm_head logits", Purpose: a fused
 *     dequant-GEMM on the packed [vocab, hidden] table, weights packed along
 *     the hidden dimension; Perf evals table: W4-g64 and W8-g128 heads at
 *     M = 1 / 32 / 256; reviewer comment items 1-2: int8 per-row heads and
 *     exact top-K rescoring from the unquantised weight.
 *   - radiance_lmhead_int4.py, quantize_int4_rows and module constants:
 *     symmetric per-group int4, QMAX 7, nibble bias 8, RTN or MSE clip-ratio
 *     search over 1.0 / 0.95 / 0.9 / 0.85 / 0.8 of amax / 7, the scale rounded
 *     to its storage dtype before q is chosen, [N, K/8] int32 packing,
 *     [N, K/G] scale table; apply(): x flattened to [M, K], optional bias.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates no device memory; scratch space is a caller buffer
 *     sized by wql_workspace_size() (wql_logits_noalloc instead uses one
 *     fixed area inside the library, see there).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy
 *     default stream).  Results are ready once the stream has reached them.
 *   - Arguments are checked on the host before anything is launched.  On any
 *     error nothing is launched and nothing is written.  The library never
 *     aborts, prints or traps; a failed CUDA launch returns WQL_ECUDA and the
 *     CUDA error text is kept for wql_last_error() (per host thread).
 *   - Row-major, densely packed tensors.  Sizes are element counts.
 *   - Empty work (m == 0 or n == 0) returns WQL_OK without launching.
 */
#ifndef WQL_H_
#define WQL_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum wql_status {
  WQL_OK = 0,
  WQL_EINVAL = 1,        /* null pointer, negative size, inconsistent args */
  WQL_EUNSUPPORTED = 2,  /* valid but not implemented here (dtype, group, K,
                            alignment) */
  WQL_ECUDA = 3,         /* a CUDA call failed; see wql_last_error() */
  WQL_EWORKSPACE = 4     /* workspace missing or smaller than required */
} wql_status;

typedef enum wql_dtype {
  WQL_F32 = 0,   /* IEEE binary32 */
  WQL_F16 = 1,   /* IEEE binary16 */
  WQL_BF16 = 2   /* bfloat16 */
} wql_dtype;

typedef enum wql_clip {
  WQL_CLIP_RTN = 0,  /* scale = amax / qmax (ratio 1.0 only) */
  WQL_CLIP_MSE = 1   /* ratios 1.0, 0.95, 0.9, 0.85, 0.8; least squared error */
} wql_clip;

/* Code format of a quantised weight (wql_weight.format). */
typedef enum wql_format {
  WQL_FMT_SYM = 0,   /* symmetric integers: int4 nibble = q + 8, or int8 q */
  WQL_FMT_E4M3 = 1,  /* bits 8, group 0: fp8 e4m3 codes, one scale per row
                        (radiance_lmhead_int4.py module docstring: the
                        per-channel fp8 head it compares against) */
  WQL_FMT_ASYM = 2   /* bits 4, group a multiple of 128: nibble = q in 0..15
                        and a zero point z per group, w ~ (q - z) * s
                        ("[CORE] Quantized lm-head Framework", the sym=False
                        lm_head model of its lm-eval table) */
} wql_format;

/* wql_weight.format = a wql_format, optionally ORed with flags: */
#define WQL_FMT_MASK 0xFF
/* WQL_WEIGHT_STATIC: no kernel that may run before a call on its stream writes
 * this weight (qweight, scales, zeros) -- it was written once, before.  The
 * decode kernel then starts copying it before the preceding kernel on the
 * stream has finished (programmatic dependent launch); X, the workspace and
 * the outputs are still touched only after it. */
#define WQL_WEIGHT_STATIC 0x100

/* A quantised lm_head weight as produced by wql_quantize() / wql_quantize_ex().
 *   bits 4: qweight is int32 [n, k/8]; word i of a row holds elements
 *           8i .. 8i+7, element 8i + j in the nibble at position
 *           p = 4*(j % 2) + j/2 (bits [4p, 4p + 4)): even elements fill bits
 *           0..15, odd elements bits 16..31, each ascending; nibble = q + 8.
 *           (The pages pack in an "ExLlama shuffle" order they do not define;
 *           this interleave is this library's format, chosen so that one
 *           mask per 16-bit half yields an adjacent element pair.)
 *   bits 8: qweight is int8 [n, k], two's complement q in [-127, 127].
 *   scales: [n, k / group] of scale_dtype, or [n, 1] when group == 0.
 *   format WQL_FMT_E4M3 (bits 8, group 0): qweight is uint8 [n, k] e4m3
 *           codes ("fn" variant: no infinities, 0x7F/0xFF NaN, largest
 *           finite 448), w ~ e4m3(q) * s[row].
 *   format WQL_FMT_ASYM (bits 4): qweight as for bits 4 with nibble = q in
 *           0..15 (no bias), zeros uint8 [n, k / group], w ~ (q - z) * s.
 * Requirements: k % 64 == 0; group is 0 or a multiple of 64 dividing k;
 * qweight 16-byte aligned; scales 2-byte aligned; n < 2^31. */
typedef struct wql_weight {
  int32_t bits;         /* 4 or 8 */
  int32_t group;        /* G (multiple of 64) or 0 = one scale per row */
  int32_t scale_dtype;  /* WQL_F16 or WQL_BF16 */
  int32_t format;       /* wql_format (WQL_FMT_SYM = 0 for the layouts above),
                           optionally | WQL_WEIGHT_STATIC */
  int64_t n;            /* vocab rows */
  int64_t k;            /* hidden size */
  const void* qweight;  /* device */
  const void* scales;   /* device */
  const void* zeros;    /* device uint8 [n, k / group] zero points 0..15
                           (WQL_FMT_ASYM), else NULL */
} wql_weight;

/* Largest top-K width supported by wql_logits / wql_topk_rescore. */
#define WQL_MAX_TOPK 16
/* Upper bound on the CTAs one wql_logits launch uses; sizes the workspace. */
#define WQL_MAX_CTAS 1024

/* Quantise and pack a dense weight (radiance_lmhead_int4.py,
 * quantize_int4_rows; int8 per the W8 rows of the Perf evals table).
 * Per group of G columns (group 0: the whole row), for each tried ratio r:
 *   s_r = RN_scale_dtype(max(fl32(amax) *f32 fl32(r / qmax), 1e-8f))
 *   q   = clamp(round_half_even(w /f32 s_r), -8 or -127, 7 or 127),
 *         and q = 0 for the whole group when s_r rounds to zero;
 * RTN keeps r = 1.0; MSE keeps the first ratio whose binary64 error
 * sum_k (q*s - w)^2 (k ascending) is strictly the smallest.
 *   w            device [n, k] of w_dtype (F32, F16 or BF16), 16-byte aligned
 *   qweight_out  device, layout of wql_weight for `bits`
 *   scales_out   device [n, k / group] (or [n]) of scale_dtype
 * Results are bit-exact with the definition above. */
wql_status wql_quantize(const void* w, int32_t w_dtype, int64_t n, int64_t k,
                        int32_t bits, int32_t group, int32_t scale_dtype,
                        int32_t clip, void* qweight_out, void* scales_out,
                        cudaStream_t stream);

/* wql_quantize with a code format (wql_format):
 *   WQL_FMT_SYM   exactly wql_quantize (zeros_out unused, may be NULL).
 *   WQL_FMT_E4M3  bits 8, group 0, clip RTN.  Per row:
 *                   s = RN_scale_dtype(max(fl32(amax) *f32 fl32(1/448), 1e-8f)),
 *                   q = RN_e4m3(clamp(w /f32 s, -448, 448)) (ties to even),
 *                 and q = 0 for the row when s rounds to zero.
 *   WQL_FMT_ASYM  bits 4, group a multiple of 128 dividing k, clip RTN.  Per
 *                 group, with lo = min(0, min w) and hi = max(0, max w):
 *                   s = RN_scale_dtype(max((hi -f32 lo) *f32 fl32(1/15), 1e-8f)),
 *                   z = clamp(rint_even(-lo /f32 s), 0, 15),
 *                   q = clamp(rint_even(w /f32 s) + z, 0, 15),
 *                 and q = z = 0 for the group when s rounds to zero;
 *                 zeros_out device uint8 [n, k / group].
 * (Neither page gives a formula for these two formats; these are the plain
 * readings: amax maps to the largest finite e4m3, and plain asymmetric
 * round-to-nearest with an integer zero point.)  Bit-exact with the
 * definitions above. */
wql_status wql_quantize_ex(const void* w, int32_t w_dtype, int64_t n, int64_t k,
                           int32_t format, int32_t bits, int32_t group,
                           int32_t scale_dtype, int32_t clip, void* qweight_out,
                           void* scales_out, void* zeros_out, cudaStream_t stream);

/* Pack nibbles (uint8 [n, k], values 0..15; higher bits are ignored) into the
 * int4 layout of wql_weight: packed_out int32 [n, k/8].  k % 8 == 0;
 * nibbles 8-byte aligned. */
wql_status wql_pack(const uint8_t* nibbles, int64_t n, int64_t k,
                    int32_t* packed_out, cudaStream_t stream);

/* Inverse of wql_pack: nibbles_out uint8 [n, k] in 0..15.  k % 8 == 0. */
wql_status wql_unpack(const int32_t* packed, int64_t n, int64_t k,
                      uint8_t* nibbles_out, cudaStream_t stream);

/* Bytes of workspace wql_logits needs for m token rows and top-K width topk
 * (n is the vocab size; the need does not grow with it).  Pure host
 * arithmetic; never touches the GPU.  The buffer must be zero-filled once
 * before its first use; every call leaves it ready for the next (except for
 * the sticky error word of a timed-out wait, see wql_debug_set_waits).
 * Calls that may run concurrently need separate workspaces. */
size_t wql_workspace_size(int64_t m, int64_t n, int32_t topk);

/* Logits of a quantised lm_head ("Fused WNA16 GEMM for tied quantized lm_head
 * logits", Purpose; radiance_lmhead_int4.py, apply()).
 *   x          device [m, k] of x_dtype (F16 or BF16), 16-byte aligned
 *   w          quantised weight (host struct; its pointers are device)
 *   bias       device [n] of x_dtype, or NULL
 *   logits_out device [m, n] of x_dtype: fp32 accumulation, then rounded to
 *              nearest-even in x_dtype
 *   topk       0 (no candidates) or 1..WQL_MAX_TOPK, topk <= n
 *   topk_idx   device int32 [m, topk] (NULL when topk == 0)
 *   topk_val   device float [m, topk]: fp32 logits, ordered by value
 *              descending, then index ascending.  For m <= 16 they are the
 *              fp32 accumulators that logits_out rounds.  For m > 16 the
 *              tensor-core kernel folds each group's scale into fp16 weights
 *              (q * s rounded to fp16); the candidates are then the rows whose
 *              rounded logit is at least the K-th largest rounded logit, and
 *              their values are recomputed in fp32 from the packed weight
 *              (exact q * x products, one fp32 sum per group, times the
 *              group's scale).  The two can differ by the folding rounding
 *              (at most 2^-11 relative per weight).
 *   workspace  device, 256-byte aligned, ws_bytes >= wql_workspace_size(m, n,
 *              topk); may be NULL when topk == 0.  A workspace that is passed
 *              is checked (size and alignment) whether or not topk is 0:
 *              WQL_EWORKSPACE otherwise.
 * The kernel is chosen from m inside the library. */
wql_status wql_logits(const void* x, int32_t x_dtype, int64_t m,
                      const wql_weight* w, const void* bias, void* logits_out,
                      int32_t topk, int32_t* topk_idx, float* topk_val,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Size of the device scratch area that wql_logits_noalloc uses: 4 MiB. */
#define WQL_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* wql_logits without a workspace argument.  The pages have no counterpart:
 * this is an interface of this library for callers that cannot provide
 * device memory -- a host program linking only this library, with no device
 * allocator of its own, or a serving loop that must not allocate after
 * start-up.  Arguments, layouts and results are those of wql_logits, except:
 *   - Scratch is one fixed area of WQL_NOALLOC_SCRATCH_BYTES per device,
 *     inside the library (reserved by the CUDA runtime when it loads the
 *     library's code on the device, and held until the process exits).  The
 *     call allocates nothing.
 *   - Every token count runs the decode kernel, in slices of at most 16
 *     token rows.  A slice's scratch need, wql_workspace_size(rows, n, topk),
 *     is at most about 2.1 MB whatever n is, so every valid call fits; a
 *     call whose slice needed more than the area would be rejected with
 *     WQL_EWORKSPACE before anything is launched.
 *   - The first call on each device does a set-up (it looks up the area's
 *     device address with that device current); it is done again after the
 *     device's context has been replaced (cudaDeviceReset, for one).  Make
 *     that first call before any stream capture begins.  A failed set-up
 *     returns WQL_ECUDA and is retried by the next call.
 *   - The area's first 256 bytes (the ticket counter of the top-K merge) are
 *     cleared on `stream` at the start of every call (one small memset
 *     before the launches).
 *   - Calls on one device share the area: calls that may be in flight at
 *     the same time (other streams, unsynchronised host threads) race and
 *     corrupt each other's outputs.  Serialise them. */
wql_status wql_logits_noalloc(const void* x, int32_t x_dtype, int64_t m,
                              const wql_weight* w, const void* bias,
                              void* logits_out, int32_t topk,
                              int32_t* topk_idx, float* topk_val,
                              cudaStream_t stream);

/* Exact top-K rescoring ("Fused WNA16 GEMM for tied quantized lm_head
 * logits", reviewer comment item 2): for every row m and each of its topk
 * candidate indices, recompute v = sum_k x[m,k] * w_ref[idx,k] (+ bias[idx])
 * with fp32 accumulation of the exact products, write logits[m, idx] =
 * RN_x_dtype(v), replace topk_val by v and re-sort the row's candidates by
 * value descending, then index ascending.
 *   x            device [m, k] of x_dtype (F16 or BF16)
 *   w_ref        device [n, k] unquantised weight, dtype == x_dtype
 *   bias         device [n] of x_dtype, or NULL
 *   topk_idx     device int32 [m, topk], each in [0, n) (in/out)
 *   topk_val     device float [m, topk] (in/out)
 *   logits_inout device [m, n] of x_dtype
 * k % 8 == 0; x and w_ref 16-byte aligned. */
wql_status wql_topk_rescore(const void* x, int32_t x_dtype, int64_t m,
                            const void* w_ref, int32_t wref_dtype, int64_t n,
                            int64_t k, const void* bias, int32_t topk,
                            int32_t* topk_idx, float* topk_val,
                            void* logits_inout, cudaStream_t stream);

/* Tied-embedding gather ("Fused WNA16 GEMM for tied quantized lm_head
 * logits", Purpose: the tied head's quantised weight also serves as the input
 * embedding, so a token's embedding row is that row of dequant(Wq)).
 *   ids        device int32 [t]; an id outside [0, n) yields a row of +0
 *   t          number of ids (0: nothing is launched)
 *   w          quantised weight (host struct; its pointers are device), the
 *              same one wql_logits reads
 *   out_dtype  WQL_F16 or WQL_BF16 (independent of the scale dtype)
 *   out        device [t, k] of out_dtype, 16-byte aligned (caller-owned):
 *              out[i, j] = RN_out(q[ids[i], j] * s[ids[i], j / group]), the
 *              product exact in fp32 and rounded once, to nearest-even
 * k % 8 == 0, k % group == 0; ids 4-byte and qweight 8-byte aligned.
 * Errors: WQL_EINVAL for NULL pointers with t > 0 or a malformed weight,
 * WQL_EUNSUPPORTED for other bit widths, dtypes, sizes or alignments;
 * asynchronous on `stream`, allocates nothing. */
wql_status wql_embed_gather(const int32_t* ids, int64_t t, const wql_weight* w,
                            int32_t out_dtype, void* out, cudaStream_t stream);

/* Static text for a status code. */
const char* wql_status_string(wql_status status);

/* Diagnostics, for tests of the timeout path.  Every wait inside the kernels
 * is bounded; a wait that runs out records bit 2 (tensor-core kernel) or 4
 * (top-K selection) in the workspace's error word (bytes 4..7, sticky until
 * the caller zeroes it), the kernel finishes without leaving copies or
 * tensor-core work in flight, and from then on the top-K outputs of every
 * call on that workspace read index -1 and value NaN.
 *   budget_cycles  SM cycles a wait of the tensor-core kernel on a ring slot
 *                  or on data may take (0: the default, about 1 s); the
 *                  waits for a CTA's own copies keep the default
 *   stall_mma      1: the tensor-core kernel's MMA warp first waits on a
 *                  barrier nothing arrives on, so that its budget runs out
 *                  and every other role's waits run out after it
 * Process-wide, for the calls launched after it; not for concurrent use.
 * (The decode kernel, m <= 16, has no waits.) */
wql_status wql_debug_set_waits(int64_t budget_cycles, int32_t stall_mma);

/* Text of the last CUDA error seen by this host thread ("" if none). */
const char* wql_last_error(void);

/* Number of kernels this process has launched through the library. */
uint64_t wql_launch_count(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* WQL_H_ */
