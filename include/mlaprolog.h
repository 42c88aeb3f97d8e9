/*
 * libmlaprolog — C ABI of the GB300 (sm_103a) MLA prolog and QKV RmsNorm-RoPE-cache operators.
 *
 * Operation definitions:
 *   - MLA prolog: MlaPrologV2 README (gitcode ops-transformer, attention/mla_prolog_v2),
 *     section 功能说明 (formulas c^Q = RmsNorm(x·W^DQ), q^C = c^Q·W^UQ, q^N = q^C·W^UK,
 *     q^R = ROPE(c^Q·W^QR), c^KV = RmsNorm(x·W^DKV) -> kv_cache, k^R = ROPE(x·W^KR) -> kr_cache),
 *     parameter table 参数说明, and shape/dtype/scenario matrix 约束说明.
 *   - QkvRmsNormRopeCache: aclnnQkvRmsNormRopeCache, "Formulas" (1) SplitVD, (2) RmsNorm,
 *     (3) RoPE half-and-half, (4) Quant, and "Other restrictions" (index semantics).
 *   - Two-phase calling pattern (size/validate, then execute on a stream):
 *     aclnnMlaPreprocessV2 / aclnnQkvRmsNormRopeCache, the GetWorkspaceSize + execute pair.
 *
 * Conventions for every call:
 *   - All tensor data pointers are DEVICE pointers of the current CUDA device, dense, row-major
 *     (C-contiguous) in the logical shape given.  Shapes use at most 4 dimensions.
 *   - The caller owns every buffer (inputs, outputs, caches, workspace, prepacked weights).  The
 *     library never allocates device memory and keeps no per-call state between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Execute calls
 *     are asynchronous on that stream; errors of the launch itself are returned, errors found by
 *     the kernels (bad cache indices, timeouts) are latched in the workspace error word and
 *     returned by mlap_check_errors().
 *   - A status other than MLAP_OK leaves outputs and caches untouched (nothing is launched) and
 *     sets a human-readable reason retrievable with mlap_last_error() (thread-local).
 *   - The kernels of a call use programmatic dependent launch: each may start while the kernel
 *     before it in the stream is finishing and read the inputs it only reads (weights, RoPE
 *     tables, norm parameters and scales, token_x outside full quant beyond 256 tokens, and qkv
 *     for qkvrnrc_execute) before it waits for that kernel; outputs, caches and the workspace
 *     are written only after that wait.  A caller's own kernel that immediately precedes a call
 *     in the stream and itself triggers programmatic dependent launch
 *     (griddepcontrol.launch_dependents) must therefore not write those inputs; any other
 *     preceding stream work (copies, kernels without that trigger) is complete before the
 *     call's first kernel starts.
 */
#ifndef MLAPROLOG_H
#define MLAPROLOG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum {
  MLAP_DTYPE_INVALID = 0,
  MLAP_DTYPE_BF16 = 1,
  MLAP_DTYPE_FP16 = 2,
  MLAP_DTYPE_FP32 = 3,
  MLAP_DTYPE_INT8 = 4,
  MLAP_DTYPE_INT64 = 5
} mlap_dtype_t;

/* A dense row-major tensor.  data == NULL means "absent" for optional parameters. */
typedef struct {
  void* data;
  int32_t dtype;     /* mlap_dtype_t */
  int32_t ndim;      /* 0..4 */
  int64_t shape[4];
} mlap_tensor_t;

typedef enum {
  MLAP_OK = 0,
  MLAP_ERR_NULL = 1,         /* a required pointer is NULL */
  MLAP_ERR_SHAPE = 2,        /* shapes disagree with the 约束说明 shape table */
  MLAP_ERR_DTYPE = 3,        /* a dtype outside the parameter table */
  MLAP_ERR_UNSUPPORTED = 4,  /* a valid combination this build does not implement */
  MLAP_ERR_WORKSPACE = 5,    /* workspace missing or smaller than the size call returned */
  MLAP_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed */
  MLAP_ERR_INDEX_RANGE = 7,  /* kernels met a cache index outside [-1, BlockNum*BlockSize) */
  MLAP_ERR_TIMEOUT = 8       /* a kernel's bounded wait ran out and the kernel returned early */
} mlap_status_t;

/* ============================================================================================ */
/* MLA prolog (MlaPrologV2 / MlaPreprocess inference prolog)                                     */
/* ============================================================================================ */

/* Symbols (约束说明): T = B*S tokens, He hidden, Hcq q-latent, Hckv kv-latent, N heads,
 * D = 128 nope head dim, Dr rope head dim (even), Nkv = 1.
 *
 * Scenarios (约束说明 scenario matrix) are selected by dtypes and optional pointers:
 *   non-quant:                   all bf16; every dequant/quant/smooth scale absent.
 *   partial quant, kv non-quant: weight_uq_qr int8 with dequant_scale_w_uq_qr (1, N*(D+Dr)) fp32
 *                                and smooth_scales_cq (1, Hcq) fp32; caches bf16.
 *   partial quant, kv quant:     as above, plus kv_cache/kr_cache int8 with quant_scale_ckv
 *                                (1, Hckv) and quant_scale_ckr (1, Dr) fp32 (value / scale,
 *                                round half to even, saturate to [-128, 127]).
 *   full quant:                  token_x int8 with dequant_scale_x (T, 1) fp32; weight_dq and
 *                                weight_dkv_kr int8 with dequant_scale_w_dq (1, Hcq) and
 *                                dequant_scale_w_dkv_kr (1, Hckv+Dr) fp32 (the integer products are
 *                                dequantised as acc * scale_x[t] * scale_w[column]); weight_uq_qr
 *                                int8 as in partial quant; kr_cache bf16.  With an int8 kv_cache
 *                                (quant_scale_ckv (1, Hckv)) the query is int8 per token and head
 *                                (scale = amax/127, written to dequant_scale_q_nope (T, N, 1));
 *                                with a bf16 kv_cache the query is bf16.
 * dequant_scale_x, dequant_scale_w_dq, dequant_scale_w_dkv_kr are reserved outside full quant
 * and must be absent (data == NULL), else MLAP_ERR_UNSUPPORTED.
 *
 * Input RmsNormQuant (aclnnMlaPreprocessV2, "Formula": RMS, RmsNorm, RmsNormQuant), optional:
 * with rms_norm_quant_gamma, _bias and _deq_scale present (all three or none), every token row
 * of token_x is replaced ahead of the down-projection by
 *     x'[t, k] = bf16((gamma[k] * x[t, k] / RMS(x[t]) + bias[k]) * deqScale[k]),
 *     RMS(x[t]) = sqrt(mean over k of x[t, k]^2 + rms_norm_quant_epsilon),
 * computed in fp32 (one value of deqScale may serve every channel).  It composes with the
 * bf16-token_x scenarios only (non-quant, partial quant); with full quant the call returns
 * MLAP_ERR_UNSUPPORTED.  token_x itself is only read. */
typedef struct {
  mlap_tensor_t token_x;            /* bf16|int8 (T, He) or (B, S, He) */
  mlap_tensor_t weight_dq;          /* prepacked W^DQ; logical shape (He, Hcq) bf16|int8 */
  mlap_tensor_t weight_uq_qr;       /* prepacked [W^UQ|W^QR]; logical (Hcq, N*(D+Dr)) bf16|int8,
                                       columns per head n: [D nope | Dr rope] */
  mlap_tensor_t weight_uk;          /* prepacked W^UK; logical (N, D, Hckv) bf16 */
  mlap_tensor_t weight_dkv_kr;      /* prepacked [W^DKV|W^KR]; logical (He, Hckv+Dr) bf16|int8 */
  mlap_tensor_t rmsnorm_gamma_cq;   /* bf16 (Hcq) */
  mlap_tensor_t rmsnorm_gamma_ckv;  /* bf16 (Hckv) */
  mlap_tensor_t rope_sin;           /* bf16 (T, Dr) or (B, S, Dr), half-and-half layout */
  mlap_tensor_t rope_cos;           /* bf16, same shape as rope_sin */
  mlap_tensor_t cache_index;        /* int64 (T) or (B, S); -1 = do not store this token */
  mlap_tensor_t kv_cache;           /* in/out (BlockNum, BlockSize, 1, Hckv) bf16|int8 */
  mlap_tensor_t kr_cache;           /* in/out (BlockNum, BlockSize, 1, Dr) bf16|int8 */
  mlap_tensor_t dequant_scale_x;        /* fp32 (T, 1) or (B*S, 1), full quant only */
  mlap_tensor_t dequant_scale_w_dq;     /* fp32 (1, Hcq), full quant only */
  mlap_tensor_t dequant_scale_w_uq_qr;  /* fp32 (1, N*(D+Dr)), partial and full quant */
  mlap_tensor_t dequant_scale_w_dkv_kr; /* fp32 (1, Hckv+Dr), full quant only */
  mlap_tensor_t quant_scale_ckv;        /* fp32 (1, Hckv), int8 kv_cache only */
  mlap_tensor_t quant_scale_ckr;        /* fp32 (1, Dr), int8 kr_cache only */
  mlap_tensor_t smooth_scales_cq;       /* fp32 (1, Hcq), partial and full quant */
  mlap_tensor_t query;              /* out (T, N, Hckv) or (B, S, N, Hckv) = q^N; bf16, or int8
                                       in full quant with an int8 kv_cache */
  mlap_tensor_t query_rope;         /* out bf16 (T, N, Dr) or (B, S, N, Dr) = q^R */
  mlap_tensor_t dequant_scale_q_nope; /* out fp32 (T, N, 1) or (B*S, N, 1) with an int8 query;
                                         otherwise may be absent and is never written */
  mlap_tensor_t rms_norm_quant_gamma;     /* optional bf16 (He): input RmsNormQuant gamma */
  mlap_tensor_t rms_norm_quant_bias;      /* optional bf16 (He): input RmsNormQuant bias */
  mlap_tensor_t rms_norm_quant_deq_scale; /* optional fp32 (He) or (1): input RmsNormQuant deqScale */
  double rmsnorm_epsilon_cq;
  double rmsnorm_epsilon_ckv;
  double rms_norm_quant_epsilon;    /* input RmsNormQuant epsilon (>= 0; read when it is on) */
  const char* cache_mode;           /* NULL or "PA_BSND" (ND paged cache); others unsupported */
} mlap_args_t;

/* Which weight a prepack call handles. */
typedef enum {
  MLAP_WEIGHT_DQ = 0,      /* (He, Hcq) */
  MLAP_WEIGHT_UQ_QR = 1,   /* (Hcq, N*(D+Dr)), bf16 or int8 */
  MLAP_WEIGHT_UK = 2,      /* (N, D, Hckv) */
  MLAP_WEIGHT_DKV_KR = 3   /* (He, Hckv+Dr) */
} mlap_weight_t;

/* Bytes of device memory a prepacked copy of `w` needs.  `w` describes the row-major weight as
 * the parameter table gives it ((k, n) for the matmul weights, 约束说明 "(k，n)"); N, D, Dr are
 * the head geometry (used by MLAP_WEIGHT_UQ_QR and MLAP_WEIGHT_UK, ignored otherwise).
 * w->data may be NULL here.  Errors: MLAP_ERR_NULL, MLAP_ERR_SHAPE, MLAP_ERR_DTYPE. */
mlap_status_t mlap_prepack_size(const mlap_tensor_t* w, int32_t which, int32_t N, int32_t D,
                                int32_t Dr, size_t* bytes);

/* Repack a row-major device weight into the layout the kernels stream (K-major rows, the
 * W^UQ|W^QR rows grouped as all nope rows then all rope rows with each RoPE pair adjacent,
 * W^UK transposed per head).  Runs once per model load, asynchronously on `stream`; `dst` is a
 * caller-owned device buffer of mlap_prepack_size() bytes and must not alias w->data.  The
 * prepacked buffer is then passed in mlap_args_t with the ORIGINAL logical shape and dtype. */
mlap_status_t mlap_prepack_weights(const mlap_tensor_t* w, int32_t which, int32_t N, int32_t D,
                                   int32_t Dr, void* dst, void* stream);

/* Phase 1 (validation and sizing; no device work, no CUDA context needed).  Checks every
 * argument against the parameter table and the shape/dtype/scenario matrix and returns the
 * workspace bytes execute needs for these shapes.  Errors: NULL, SHAPE, DTYPE, UNSUPPORTED. */
mlap_status_t mlap_get_workspace_size(const mlap_args_t* args, size_t* bytes);

/* Zero the workspace's error word (its first 256 bytes).  Call once after allocating a workspace (or
 * cudaMemset the first 256 bytes to 0).  Asynchronous on `stream`. */
mlap_status_t mlap_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Phase 2: run the prolog on `stream`.  Re-validates the arguments (same errors as phase 1),
 * plus MLAP_ERR_WORKSPACE if workspace_bytes is below the phase-1 size, MLAP_ERR_CUDA if a launch
 * fails.  T == 0: returns MLAP_OK with nothing launched.  BlockNum*BlockSize == 0: outputs are
 * computed and the caches are not touched.  Writes query, query_rope and the cache rows named by
 * cache_index; every other cache row stays bit-identical.  Indices outside [-1, BlockNum*
 * BlockSize) are skipped and latched (see mlap_check_errors).  Indices must be unique (caller
 * contract); with repeats the row stored in that slot is unspecified.  Results are bitwise
 * deterministic for a given device and shapes.  The workspace must not be shared by calls that
 * may run concurrently. */
mlap_status_t mlap_execute(const mlap_args_t* args, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Synchronise `stream`, read and clear the workspace error word.  Returns MLAP_OK,
 * MLAP_ERR_INDEX_RANGE or MLAP_ERR_TIMEOUT (index errors take precedence), or MLAP_ERR_CUDA. */
mlap_status_t mlap_check_errors(void* workspace, void* stream);

/* Exercise the kernels' failure path: launches one kernel that waits, with the same bounded
 * wait as every kernel of the library, on a barrier that nothing completes.  The wait gives up
 * after its limit (about 2 s), and the kernel latches the timeout bit in the workspace error
 * word, so a following mlap_check_errors returns MLAP_ERR_TIMEOUT (and clears the word, as it
 * always does).  Nothing faults or hangs.
 * Asynchronous on `stream`.  Errors: MLAP_ERR_NULL, MLAP_ERR_WORKSPACE (fewer than 256 bytes),
 * MLAP_ERR_CUDA. */
mlap_status_t mlap_selftest_bounded_wait(void* workspace, size_t workspace_bytes, void* stream);

/* ============================================================================================ */
/* QkvRmsNormRopeCache (aclnnQkvRmsNormRopeCache)                                                */
/* ============================================================================================ */

/* qkv (B, S, (Nq+Nk+Nv)*D) or (T, (Nq+Nk+Nv)*D), fp16 or bf16, D = 128 (the page: "Currently,
 * only 128 is supported"), Nk == Nv.  Per token:
 *   q, k, v = SplitVD(qkv);  q, k <- RoPE_half_and_half(RmsNorm(., gamma, epsilon), cos, sin);
 *   q_out = q;  k_cache[index] = Quant(k);  v_cache[index] = Quant(v)
 * Quant ("Formulas" (4)): none when k_scale/v_scale are absent (caches have qkv's dtype);
 * symmetric (value / scale) when the scales are present; asymmetric (value / scale + offset)
 * when k_offset/v_offset are present too; the int8 code rounds half to even and saturates to
 * [-128,127].  It is computed as value * fp32(1/scale) (+ offset) in fp32, so a code can differ
 * from the exact quotient's by one near a rounding tie.  Scales must be nonzero (caller
 * contract, "Other restrictions").
 * Optional outputs (the API function's qBeforeQuant / kBeforeQuant / vBeforeQuant): the tensors
 * that enter Quant, dense in token order (one row per token, including index -1), in qkv's dtype:
 * q after RoPE (equal to q_out), k after RoPE, v as split. */
typedef struct {
  mlap_tensor_t qkv;       /* fp16|bf16 */
  mlap_tensor_t gamma_q;   /* (D), dtype of qkv, shared by all q heads */
  mlap_tensor_t gamma_k;   /* (D), dtype of qkv, shared by all k heads */
  mlap_tensor_t cos;       /* (T, D) or (B, S, D), dtype of qkv, shared by all heads */
  mlap_tensor_t sin;       /* same as cos */
  mlap_tensor_t index;     /* int64 (T) or (B, S); values in [-1, BlockNum*BlockSize), unique */
  mlap_tensor_t k_cache;   /* in/out (BlockNum, BlockSize, Nk, D) int8 or dtype of qkv */
  mlap_tensor_t v_cache;   /* in/out (BlockNum, BlockSize, Nv, D), same dtype as k_cache */
  mlap_tensor_t k_scale;   /* fp32 (Nk, D) or absent */
  mlap_tensor_t v_scale;   /* fp32 (Nv, D) or absent */
  mlap_tensor_t k_offset;  /* fp32 (Nk, D) or absent: asymmetric quant (needs the scales) */
  mlap_tensor_t v_offset;  /* fp32 (Nv, D), present exactly when k_offset is */
  mlap_tensor_t q_out;     /* out (T, Nq, D) or (B, S, Nq, D), dtype of qkv */
  mlap_tensor_t q_before_quant;  /* optional out, same layout and dtype as q_out */
  mlap_tensor_t k_before_quant;  /* optional out (T, Nk, D) or (B, S, Nk, D), dtype of qkv */
  mlap_tensor_t v_before_quant;  /* optional out (T, Nv, D) or (B, S, Nv, D), dtype of qkv */
  int32_t Nq, Nk, Nv;
  double epsilon;
  const char* cache_mode;  /* NULL or "PA_BSND"; "PA_NZ" is unsupported */
} qkvrnrc_args_t;

/* Phase 1: validate and size.  BlockNum must satisfy BlockNum >= ceil(S/BlockSize)*B
 * ("Input shape restrictions").  Errors: NULL, SHAPE, DTYPE, UNSUPPORTED. */
mlap_status_t qkvrnrc_get_workspace_size(const qkvrnrc_args_t* args, size_t* bytes);

/* Phase 2: run on `stream`.  Same workspace conventions as mlap_execute (initialise once with
 * mlap_workspace_init; read index errors with mlap_check_errors). */
mlap_status_t qkvrnrc_execute(const qkvrnrc_args_t* args, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ============================================================================================ */
/* Utilities                                                                                     */
/* ============================================================================================ */

/* Static string naming a status code. */
const char* mlap_status_string(mlap_status_t status);

/* Reason for the last non-OK status returned on this thread ("" if none). */
const char* mlap_last_error(void);

/* Execution stamps, for profiling a call whose kernels overlap (programmatic dependent launch
 * lets each kernel start while the one before it finishes, so events between the launches would
 * change what they measure).  mlap_execute_stamped is mlap_execute launching the same kernels in
 * the same way, each of which also records %globaltimer readings (ns) in `stamps`, a
 * caller-owned device buffer of MLAP_STAMP_KERNELS * MLAP_STAMP_BLOCK uint64 words, 8-byte
 * aligned, that the caller zeroes before the call (the call itself adds no work to the stream,
 * so a stamped call pipelines with its neighbours exactly as an unstamped one).  Each kernel
 * writes the slot of its kind:
 *   slot k starts at word k * MLAP_STAMP_BLOCK;
 *   word 0: bitwise complement of the earliest CTA start, word 1: the latest CTA end;
 *   words 4 + 4c + i for CTA c < MLAP_STAMP_CTAS: i = 0 start, 1 the wait on the preceding
 *   kernel returned, 2 the main loop's results ready (accumulator or reduction), 3 end.
 * A slot whose kernel did not run stays zero.  Slots: MLAP_STAMP_DOWN down-projection;
 * MLAP_STAMP_NORM RmsNorm/RoPE/quant/scatter; MLAP_STAMP_UP up-projection, or the fused
 * up-projection and absorb where one kernel runs both (decode: T <= 128, N >= 16, D = 128,
 * Dr = 64, Hckv <= 512 and a multiple of 32); MLAP_STAMP_ABSORB the separate absorb;
 * MLAP_STAMP_QKV the QkvRmsNormRopeCache kernel (qkvrnrc_execute_stamped).  The small helper
 * kernels (input RmsNormQuant, full-quant token_x widening beyond 256 tokens, int8 query
 * quantisation) record nothing.
 * Same errors as the execute calls, plus MLAP_ERR_NULL for a NULL `stamps`.  Stamps are
 * profiling aids with the resolution of %globaltimer; nothing in the results depends on them. */
#define MLAP_STAMP_KERNELS 5
#define MLAP_STAMP_BLOCK 1024
#define MLAP_STAMP_CTAS 255
#define MLAP_STAMP_DOWN 0
#define MLAP_STAMP_NORM 1
#define MLAP_STAMP_UP 2
#define MLAP_STAMP_ABSORB 3
#define MLAP_STAMP_QKV 4
mlap_status_t mlap_execute_stamped(const mlap_args_t* args, void* workspace,
                                   size_t workspace_bytes, void* stream, uint64_t* stamps);
mlap_status_t qkvrnrc_execute_stamped(const qkvrnrc_args_t* args, void* workspace,
                                      size_t workspace_bytes, void* stream, uint64_t* stamps);

/* ============================================================================================ */
/* Allocation-free MLA prolog                                                                    */
/* ============================================================================================ */

/* The operator pages have no counterpart to this call: it exists for callers that cannot
 * allocate device memory or pass a workspace, such as a plugin whose host framework owns every
 * device buffer and only hands over the tensors it manages, a latency-critical loop that cannot
 * pay cudaMalloc's implicit device synchronisation, or a plain C caller without a device
 * allocator.
 *
 * Same arguments, validation, kernels and results as mlap_execute, but no workspace: the scratch
 * lives in a static device array of MLAP_NO_ALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that uses this call keeps until the process exits.  The caller still passes all inputs and
 * outputs.  The call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *   - Shapes whose workspace (mlap_get_workspace_size) exceeds MLAP_NO_ALLOC_SCRATCH_BYTES are
 *     rejected with MLAP_ERR_WORKSPACE before any device work.  With the decode shapes
 *     (He 7168, Hcq 1536, Hckv 512, N 128, D 128, Dr 64) in the non-quant scenario without
 *     the input RmsNormQuant (which adds T * He * 2 bytes, as full quant does beyond 256
 *     tokens), calls with T <= 147 or 257 <= T <= 568 tokens fit (up to 256 tokens the
 *     down-projection keeps up to 16 K-split partials, above that one).
 *   - Every call looks up the array's device address on the current device (the first lookup on
 *     a device may load the library's device code there); make the first call on each device
 *     before any stream capture on it.
 *   - Every call on a device shares the one array and clears its error word first; calls that
 *     may overlap on the GPU (different streams, or other threads) race on it and must be
 *     serialised by the caller.  Kernel-detected cache-index errors are skipped on the device
 *     and are not reported by this call (use mlap_execute + mlap_check_errors to see them). */
#define MLAP_NO_ALLOC_SCRATCH_BYTES (24u * 1024u * 1024u)
mlap_status_t mlap_execute_no_alloc(const mlap_args_t* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLAPROLOG_H */
