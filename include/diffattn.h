/*
 * diffattn.h — C ABI of libdiffattn.so: causal multi-head differential
 * attention on one GB300 (sm_103a).
 *
 * The operation, as the source pages define it:
 *
 *   DiffAttn(X) = (softmax(Q1 K1^T / sqrt(d)) - lambda * softmax(Q2 K2^T / sqrt(d))) V
 *   lambda      = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
 *   lambda_init = 0.8 - 0.6 * exp(-0.3 * (l - 1))          (l = 1-based layer index)
 *   y_head      = RMSNorm(DiffAttn_head) * (1 - lambda_init)
 *
 * "Differential Transformer: Transformer que cancela ruído de atenção"
 * (pt.news.hada.io), sections "Como a atenção diferencial funciona" and
 * "Estrutura multi-head e arquitetura completa"; the causal mask (M_ij = 0 for
 * i >= j, -inf for i < j) from "A Simple Principle From Noise-Cancelling
 * Headphones Supercharges Transformers Like Never Before" (intoai.pub),
 * section "A Deeper Dive Into Attention Calculations".
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer; the library allocates no device memory and
 *    never synchronises, except diffattn_read_error (documented there).
 *  - All pointers are device pointers unless stated otherwise. Work is
 *    enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *    Some kernels (the GEMMs, the wide-head attention, add+RMSNorm, the
 *    backward's key side) are programmatic dependent launches: their CTAs may
 *    start their setup while the previous kernel on the stream finishes, but
 *    they read nothing and complete nothing before it has completed, so stream
 *    order holds as for ordinary launches (also under CUDA-graph capture).
 *  - Every call returns a diffattn_status; nothing throws across the ABI.
 *    Shapes, dtypes, alignment and strides are checked on the host before any
 *    launch (DIFFATTN_ERR_INVALID_ARG); shape families without a kernel give
 *    DIFFATTN_ERR_UNSUPPORTED; a failed launch gives DIFFATTN_ERR_CUDA.
 *  - Kernels never spin without bound. A wait that exceeds its iteration cap
 *    records a code in the workspace's error word and the kernel returns;
 *    diffattn_read_error reports it as DIFFATTN_ERR_TIMEOUT.
 *  - Softmax scale is 1/sqrt(d), d = the width of one query/key half.
 *  - bf16 means bfloat16 and f16 IEEE binary16, each stored in 2 bytes; f32
 *    means IEEE binary32.
 */
#ifndef DIFFATTN_H
#define DIFFATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DIFFATTN_OK = 0,
    DIFFATTN_ERR_INVALID_ARG = 1,  /* bad pointer, shape, stride, alignment or dtype */
    DIFFATTN_ERR_UNSUPPORTED = 2,  /* valid arguments, but no kernel for this (dtype, d, Dv) */
    DIFFATTN_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than the size query returns */
    DIFFATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    DIFFATTN_ERR_TIMEOUT = 5       /* a device-side bounded wait gave up (see diffattn_read_error) */
} diffattn_status;

typedef enum { DIFFATTN_F32 = 0, DIFFATTN_BF16 = 1, DIFFATTN_F16 = 2 } diffattn_dtype;

/* A 4-D [B, H, rows, width] operand whose last dimension is contiguous.
 * Strides are in ELEMENTS. ptr and every stride times the element size must be
 * multiples of 16 bytes. */
typedef struct {
    const void* ptr;
    int64_t stride_b;
    int64_t stride_h;
    int64_t stride_n;
} diffattn_tensor;

/* Human-readable name of a status code (static storage). */
const char* diffattn_status_string(int status);

/*
 * diffattn_lambda — the lambda reparameterisation, on the host.
 *   lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
 *   lambda_init = 0.8 - 0.6 * exp(-0.3 * (layer - 1))   if lambda_init_override < 0
 *   lambda_init = lambda_init_override                   otherwise (the constant-0.8 ablation)
 * Source: "Differential Transformer: Transformer que cancela ruído de atenção",
 * section "Como a atenção diferencial funciona"; "Tag: Attention Mechanism"
 * (priorstack.com), section "Cancelling Context Noise Through Attention Map
 * Subtraction". One lambda serves every head of a layer (section "Estrutura
 * multi-head e arquitetura completa").
 *
 * lq1, lk1, lq2, lk2: HOST pointers to d floats each. layer: 1-based.
 * Computed in double, returned rounded to float in *lambda_out and
 * *lambda_init_out (host pointers). INVALID_ARG on NULL pointers, d < 1,
 * layer < 1 (when the schedule is used) or a non-finite result.
 */
diffattn_status diffattn_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                                int d, int layer, float lambda_init_override,
                                float* lambda_out, float* lambda_init_out);

/*
 * diffattn_fwd — fused causal prefill: both softmax maps, their lambda-weighted
 * difference times V, the per-head RMSNorm and the (1 - lambda_init) scale.
 * Source: the DiffAttn formula ("Como a atenção diferencial funciona") and the
 * per-head normalisation ("Estrutura multi-head e arquitetura completa") of
 * "Differential Transformer: Transformer que cancela ruído de atenção"; causal
 * mask from "A Deeper Dive Into Attention Calculations" (intoai.pub page).
 *
 * q1, q2, k1, k2: [B, H, N, d]; v: [B, H, N, Dv]; all of dtype in_dtype
 *   (f32, bf16 or f16).
 *   Query row i sits at position i and, when causal != 0, sees keys 0..i.
 *   With causal == 0 every row sees all N keys.
 * out: [B, N, H, Dv] contiguous, dtype out_dtype (tokens outermost, heads
 *   concatenated on channels: the layout W_O multiplies).
 * norm_weight: NULL (weight 1) or [Dv] f32, the RMSNorm gain.
 * y = o / sqrt(mean_Dv(o^2) + eps) * norm_weight * (1 - lambda_init).
 * Supported: in_dtype f32 with d <= 128 (multiple of 4) and Dv <= 256
 * (multiple of 32), fp32 arithmetic throughout; in_dtype bf16 or f16 with
 * (d, Dv) = (64, 128) or (128, 256), tcgen05 tensor-core kernels with fp32
 * accumulation (the probability tile P is rounded to the operand type for the
 * P.V product). out_dtype f32 or bf16 for every in_dtype; f16 as well for bf16
 * and f16 inputs.
 * Range: scores, running maxima, row sums and accumulators are fp32 and P is
 *   kept below 2^8 (the running maximum is refreshed whenever a row's maximum
 *   grows by more than 8 in log2 units). The exponent S log2(e)/sqrt(d) - max is
 *   one fused multiply-add whose rounding residual grows with the scores: up to
 *   half an fp32 ulp of the row maximum, which stays below 1 for scaled scores
 *   |S log2(e)/sqrt(d)| < 2^24 and below the 16-bit P range for < 2^28. Scores
 *   beyond 2^28 (far past one-hot: a softmax saturates long before) are outside
 *   the supported range and may give a non-finite row. Precision: the output's
 *   sensitivity to the rounding of Q and K grows with the scores' magnitude, as
 *   for any softmax. y is RMS-normalised (|y| <= sqrt(Dv) * |weight| *
 *   |1 - lambda_init|), so an f16 out_dtype cannot overflow.
 * B, H or N equal to 0: nothing to do, returns DIFFATTN_OK.
 * workspace: at least diffattn_fwd_workspace_size() bytes, 256-byte aligned;
 *   its first 4 bytes are the device error word, which must be zero before the
 *   first call (diffattn_read_error re-zeroes it); the rest needs no
 *   initialisation.
 */
diffattn_status diffattn_fwd(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                             diffattn_tensor v, void* out, const float* norm_weight,
                             int B, int H, int N, int d, int Dv, int causal,
                             float lambda, float lambda_init, float eps,
                             int in_dtype, int out_dtype,
                             void* workspace, size_t workspace_bytes, void* stream);

diffattn_status diffattn_fwd_workspace_size(int B, int H, int N, int d, int Dv, size_t* bytes);

/*
 * diffattn_decode — one new query token per sequence against its KV cache,
 * split over the cache length and merged (both softmax states are merged
 * exactly, then combined, normalised and scaled as in diffattn_fwd).
 * Source: as diffattn_fwd, applied to the last row of each sequence; the KV
 * cache read at every decoding step is the cost "Tag: Attention Mechanism"
 * (priorstack.com), article "Multi-Head Latent Attention: Scaling LLM Serving
 * Throughput via Low-Rank KV Compression", describes.
 *
 * q1, q2: [B, H, d] contiguous bf16 (the new token's two query halves).
 * k1_cache, k2_cache: [B, H, Lmax, d] bf16; v_cache: [B, H, Lmax, Dv] bf16.
 * seq_lens: device int32 [B], 1 <= seq_lens[b] <= L, or NULL (every sequence has
 *   length L). Values are clamped to [0, L] on the device; a length of 0 has
 *   no keys and yields NaN for that sequence. The query is the last of its sequence's seq_lens[b] tokens (its
 *   own K/V already appended) and sees cache entries 0..seq_lens[b]-1.
 * L: the cache capacity used (<= the allocated Lmax; entries beyond are not read).
 * out: [B, H, Dv] contiguous, out_dtype.
 * num_splits: 0 = choose automatically; otherwise 1..256 key-range splits.
 * Supported: bf16 with (d, Dv) = (64, 128) or (128, 256).
 * workspace: at least diffattn_decode_workspace_size() bytes, 256-byte aligned,
 *   for the error word (first 4 bytes, zero before the first call, as for
 *   diffattn_fwd) and the split partial states (no initialisation needed).
 * B or H equal to 0: returns DIFFATTN_OK without launching.
 */
diffattn_status diffattn_decode(const void* q1, const void* q2,
                                diffattn_tensor k1_cache, diffattn_tensor k2_cache, diffattn_tensor v_cache,
                                const int32_t* seq_lens, int L,
                                void* out, const float* norm_weight,
                                int B, int H, int d, int Dv, float lambda, float lambda_init, float eps,
                                int num_splits, int out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for diffattn_decode with these sizes; num_splits as above. Also
 * large enough for diffattn_decode_paged and diffattn_decode_paged_fp8 with the
 * same sizes (the fp8 decode may choose more splits; the larger count is used). */
diffattn_status diffattn_decode_workspace_size(int B, int H, int L, int d, int Dv, int num_splits, size_t* bytes);

/*
 * diffattn_decode_noalloc — diffattn_decode for callers that cannot allocate
 * device memory: the same kernels and results, but the split partial states
 * and the error word live in a scratch array inside the library instead of a
 * caller-provided workspace. The pages have no counterpart to this entry
 * point; it exists for hosts such as plugin or embedded runtimes that hand the
 * code pre-allocated inputs and outputs but forbid cudaMalloc (and therefore
 * cannot supply a workspace).
 *
 * Arguments are those of diffattn_decode without workspace/workspace_bytes.
 * Scratch: a file-scope device array of DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES
 * (8 MiB) that every GPU loading the library holds until process exit. Calls
 * whose partial states need more (the split states diffattn_decode would use for
 * the same arguments larger than the limit) are rejected with
 * DIFFATTN_ERR_WORKSPACE before anything is launched.
 * Set-up: every call looks up the array's device address in the current
 * device's context (cudaGetSymbolAddress). The first lookup on a device loads
 * the library's device code there, so make the first call on each device before
 * any stream capture. Looking the address up each time keeps it right after a
 * device reset, which reloads the code and may move the array. No call
 * allocates or frees device memory.
 * Errors: the arguments are checked exactly as diffattn_decode checks them,
 * before the scratch is touched, so a rejected call writes nothing to it.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; the error word is cleared (cudaMemsetAsync on `stream`) at
 * the start of each call. Calls that overlap on the GPU (different streams
 * without ordering) race on the array and give undefined results. A device-side
 * wait that gives up is recorded in the array's error word: read it with
 * diffattn_decode_noalloc_read_error before the next call clears it.
 */
#define DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
diffattn_status diffattn_decode_noalloc(const void* q1, const void* q2,
                                        diffattn_tensor k1_cache, diffattn_tensor k2_cache, diffattn_tensor v_cache,
                                        const int32_t* seq_lens, int L,
                                        void* out, const float* norm_weight,
                                        int B, int H, int d, int Dv, float lambda, float lambda_init, float eps,
                                        int num_splits, int out_dtype, void* stream);

/* diffattn_decode_noalloc_read_error — host only: reads the error word of the
 * no-allocation decode's scratch on the current device, after synchronising
 * `stream`, and clears it when it is set, like diffattn_read_error does for a
 * workspace. *device_code receives the raw device code (0 = no error).
 * Returns DIFFATTN_OK when it was 0, DIFFATTN_ERR_TIMEOUT when a device-side
 * wait gave up, DIFFATTN_ERR_CUDA if the copy or the address lookup failed,
 * DIFFATTN_ERR_INVALID_ARG if device_code is NULL. No counterpart in the pages. */
diffattn_status diffattn_decode_noalloc_read_error(void* stream, int32_t* device_code);

/*
 * diffattn_decode_paged — diffattn_decode against a paged KV cache, with query
 * heads optionally sharing KV heads (grouped-query attention). Same
 * computation, kernels and split geometry as diffattn_decode; only where each
 * key's K1, K2 and V rows are read from changes. The pages name the KV cache
 * read at every decoding step as the decode cost ("Tag: Attention Mechanism",
 * priorstack.com, Multi-Head Latent Attention article) and mention GQA
 * (hada page, Hacker News discussion); paging and sharing are serving layouts,
 * not part of the method.
 *
 * k1_pages, k2_pages: [num_pages, H_kv, 64, d] bf16; v_pages: [num_pages, H_kv,
 *   64, Dv] bf16 (a page holds 64 consecutive tokens of one sequence for every
 *   KV head; stride_b of the tensors is the page stride, stride_n the token
 *   stride within a page; last dimension contiguous).
 * block_table: device int32 [B, max_pages]; block_table[b * max_pages + i] is
 *   the physical page holding tokens 64i .. 64i+63 of sequence b, for every i
 *   < ceil(seq_lens[b] / 64). Entries outside [0, num_pages) are not checked
 *   on the device: they read zeros (the copy engine fills out-of-range tiles)
 *   and give a wrong result, never a memory fault.
 * seq_lens: device int32 [B], required; clamped to [0, L] as in diffattn_decode.
 * L: the largest sequence length (<= 64 * max_pages); sizes the split geometry.
 * H: query heads; kv_group >= 1 divides H, and query head h reads KV head
 *   h / kv_group (H_kv = H / kv_group).
 * Other arguments, the workspace (diffattn_decode_workspace_size with the same
 * B, H, L, d, Dv, num_splits) and errors: as diffattn_decode.
 */
diffattn_status diffattn_decode_paged(const void* q1, const void* q2,
                                      diffattn_tensor k1_pages, diffattn_tensor k2_pages, diffattn_tensor v_pages,
                                      const int32_t* block_table, int max_pages, int num_pages,
                                      const int32_t* seq_lens, int L,
                                      void* out, const float* norm_weight,
                                      int B, int H, int kv_group, int d, int Dv,
                                      float lambda, float lambda_init, float eps,
                                      int num_splits, int out_dtype,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * diffattn_kv_append_paged — writes each sequence's new token into a paged KV
 * cache (the layout of diffattn_decode_paged) before the decode step that
 * attends to it: for every sequence b and KV head h, the rows k1_new[b, h],
 * k2_new[b, h] and v_new[b, h] go to row pos % 64 of page
 * block_table[b * max_pages + pos / 64], where pos = seq_lens[b] - 1 (the new
 * token is the last of its sequence, as in the decode calls). A plain copy,
 * bit-exact; a sequence whose position or page falls outside the table or the
 * pool is skipped.
 *
 * k1_new, k2_new: [B, H_kv, d] bf16, v_new: [B, H_kv, Dv] bf16, contiguous and
 *   16-byte aligned. k1_pages and k2_pages must share their strides.
 * block_table, seq_lens: device int32, as for diffattn_decode_paged.
 * d and Dv multiples of 8. B or H_kv equal to 0: returns DIFFATTN_OK.
 */
diffattn_status diffattn_kv_append_paged(const void* k1_new, const void* k2_new, const void* v_new,
                                         diffattn_tensor k1_pages, diffattn_tensor k2_pages, diffattn_tensor v_pages,
                                         const int32_t* block_table, int max_pages, int num_pages,
                                         const int32_t* seq_lens, int B, int H_kv, int d, int Dv, void* stream);

/*
 * diffattn_decode_paged_fp8 — diffattn_decode_paged against a paged cache of
 * fp8 e4m3 values with one scale per tensor: cached K1 = k1_pages * k1_scale,
 * K2 = k2_pages * k2_scale, V = v_pages * v_scale. Half the bytes of the bf16
 * cache for the HBM-bound decode. The pages point to lower-bit quantization as
 * a use of differential attention's smaller activation outliers ("Differential
 * Transformer: Transformer que cancela ruído de atenção", section "Resultados
 * experimentais e efeitos de aplicação"). Arithmetic is fp32 on the
 * dequantized values (the query stays bf16), so the result is the decode of
 * the dequantized cache.
 *
 * k1_pages, k2_pages: [num_pages, H_kv, 64, d] e4m3 bytes; v_pages: [num_pages,
 *   H_kv, 64, Dv] e4m3 bytes (strides in elements = bytes, multiples of 16).
 * k1_scale, k2_scale, v_scale: finite and > 0 (else INVALID_ARG).
 * Other arguments, the workspace and errors: as diffattn_decode_paged.
 */
diffattn_status diffattn_decode_paged_fp8(const void* q1, const void* q2,
                                          diffattn_tensor k1_pages, diffattn_tensor k2_pages, diffattn_tensor v_pages,
                                          const int32_t* block_table, int max_pages, int num_pages,
                                          const int32_t* seq_lens, int L,
                                          void* out, const float* norm_weight,
                                          int B, int H, int kv_group, int d, int Dv,
                                          float lambda, float lambda_init, float eps,
                                          float k1_scale, float k2_scale, float v_scale,
                                          int num_splits, int out_dtype,
                                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * diffattn_kv_append_paged_fp8 — diffattn_kv_append_paged into fp8 e4m3 pages:
 * each value x of the bf16 rows k1_new, k2_new, v_new is stored as
 * e4m3(x / scale) (x / scale rounded to fp32, then to the nearest e4m3 value,
 * ties to even, saturating at +-448). Scales finite and > 0; other arguments
 * and errors as diffattn_kv_append_paged (page strides in bytes).
 */
diffattn_status diffattn_kv_append_paged_fp8(const void* k1_new, const void* k2_new, const void* v_new,
                                             diffattn_tensor k1_pages, diffattn_tensor k2_pages,
                                             diffattn_tensor v_pages, const int32_t* block_table, int max_pages,
                                             int num_pages, const int32_t* seq_lens, int B, int H_kv, int d, int Dv,
                                             float k1_scale, float k2_scale, float v_scale, void* stream);

/*
 * diffattn_bwd — gradients of diffattn_fwd (the backward pass). The pages train
 * DIFF Transformers ("Differential Transformer: Transformer que cancela ruído
 * de atenção", section "Eficiência e estabilidade de treinamento") but print no
 * gradient; this computes the chain rule of the forward definition. With
 * P_m = softmax(Q_m K_m^T / sqrt d + M), A = P1 - lambda P2, O = A V and
 * y = O / sqrt(mean(O^2) + eps) * w * (1 - lambda_init):
 *   dO = (g - n mean(g n)) / r with n = O / r, g = dy w (1 - lambda_init);
 *   dV = A^T dO; dA = dO V^T; dlambda = -sum(dA P2);
 *   dS1 = P1 (dA - rowsum(P1 dA)); dS2 = P2 (-lambda dA - rowsum(-lambda P2 dA));
 *   dQ_m = dS_m K_m / sqrt d; dK_m = dS_m^T Q_m / sqrt d; dw = sum_rows dy n (1 - lambda_init).
 * lambda_init is a constant of the layer and has no gradient.
 *
 * q1..v, norm_weight, B, H, N, d, Dv, causal, lambda, lambda_init, eps,
 *   in_dtype: as for diffattn_fwd (in_dtype f32, bf16 or f16).
 * dy: [B, N, H, Dv] contiguous, in_dtype — the gradient with respect to the
 *   forward's output, in the forward's output layout.
 * dq1, dq2, dk1, dk2: [B, H, N, d] contiguous f32; dv: [B, H, N, Dv] contiguous
 *   f32 (written, not accumulated).
 * dlambda: device f32[1], the sum over every head (lambda is shared by the
 *   layer's heads); chain it to the lambda vectors with diffattn_lambda_bwd.
 * dnorm_weight: device f32[Dv] or NULL — the gradient with respect to the
 *   RMSNorm gain (of a unit gain when norm_weight is NULL).
 * d and Dv multiples of 32 with d <= 128 and Dv <= 256 (else UNSUPPORTED).
 * Every pointer 16-byte aligned. Two paths, chosen by shape and type:
 *   bf16 or f16 with (d, Dv) = (64, 128): tcgen05 tensor cores. The forward is
 *     re-run with an epilogue that leaves dO (rounded to in_dtype), the per-row
 *     log-sum-exps, D1 = dO.(P1 V), D2 = -lambda dO.(P2 V) and per-tile partial
 *     sums of dlambda and dw; a key-side kernel forms dV and dK1, dK2 and a
 *     query-side kernel dQ1, dQ2, both from S, P and dA recomputed on the tensor
 *     cores with fp32 accumulation. dO, A and dS1, dS2 are rounded to in_dtype
 *     as the left operands of their products (like P in the forward): about
 *     2.5e-3 relative RMS per gradient for bf16 and 3e-4 for f16.
 *   otherwise (f32 inputs, other widths): fp32 arithmetic on the CUDA cores.
 * Results do not depend on scheduling (no atomics): every gradient row is
 * written by one CTA and the partial sums are added in a fixed order.
 * Streams (tensor-core path): the query-side kernel and the reduction run on a
 * side stream the library owns (one per device, created on first use), forked
 * from `stream` after the preparation and joined back into it before the call
 * returns, so work enqueued on `stream` afterwards sees every output. Concurrent
 * calls from several host threads are serialised around the shared side stream.
 * B, H or N equal to 0: DIFFATTN_OK.
 * workspace: diffattn_bwd_workspace_size() bytes, 256-byte aligned.
 */
diffattn_status diffattn_bwd(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                             diffattn_tensor v, const void* dy, const float* norm_weight,
                             int B, int H, int N, int d, int Dv, int causal,
                             float lambda, float lambda_init, float eps, int in_dtype,
                             float* dq1, float* dq2, float* dk1, float* dk2, float* dv,
                             float* dlambda, float* dnorm_weight,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes diffattn_bwd needs: the control block, dO and four per-row
 * statistics (dO in f32, or in the 16-bit input type on the tensor-core path),
 * and per-block partial sums of dlambda and dw. */
diffattn_status diffattn_bwd_workspace_size(int B, int H, int N, int d, int Dv, size_t* bytes);

/*
 * Training pair: a forward that also saves the state the backward starts from,
 * and the backward that starts from it instead of re-running the forward.
 *
 * diffattn_fwd_train — diffattn_fwd (same arguments, same output, bit for bit)
 * that also writes into `saved` what the backward needs of the forward once its
 * last PV products finished: per row, x = O1/l1 - lambda O2/l2, the output before
 * the norm (f32 [B, H, N, Dv], the forward's own values); map 2's attention output
 * O2/l2 = softmax_2 V rounded once to the operand type ([B, H, N, Dv], 16-bit; the
 * backward forms O1/l1 = x + lambda O2/l2); and each map's log-sum-exp in base 2 of
 * the scaled scores, L_m = max_m + log2(l_m) = log2 sum_j exp2(S_m log2(e)/sqrt(d))
 * (f32 [B, H, N, 2]). Tensor-core path only: bf16 or f16 with (d, Dv) = (64, 128)
 * (else DIFFATTN_ERR_UNSUPPORTED); it always runs the per-tile kernel.
 * saved: device, diffattn_train_saved_size() bytes, 256-byte aligned, owned by
 *   the caller; the contents are meant only for diffattn_bwd_saved with the same
 *   q1..v, norm_weight, shapes, causal, lambda, lambda_init, eps and in_dtype.
 *
 * diffattn_bwd_saved — diffattn_bwd (same arguments and outputs) from `saved`:
 * its preparation (one CUDA-core pass over the rows, bandwidth-bound) reads x,
 * O2/l2 and L_m instead of recomputing the scores, softmaxes and PV products, then
 * the same key-side, query-side and reduction kernels run. The gradients agree with
 * diffattn_bwd's to rounding: O2/l2 carries one rounding to the operand type (it
 * enters D1 and D2 only; the norm's x is exact) and the per-row sums (the norm, D1,
 * D2) are added in another fp32 order.
 * Deterministic. Same support as diffattn_fwd_train; workspace as for
 * diffattn_bwd.
 */
diffattn_status diffattn_train_saved_size(int B, int H, int N, int Dv, size_t* bytes);
diffattn_status diffattn_fwd_train(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                                   diffattn_tensor v, void* out, const float* norm_weight,
                                   int B, int H, int N, int d, int Dv, int causal,
                                   float lambda, float lambda_init, float eps, int in_dtype, int out_dtype,
                                   void* saved, size_t saved_bytes,
                                   void* workspace, size_t workspace_bytes, void* stream);
diffattn_status diffattn_bwd_saved(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                                   diffattn_tensor v, const void* dy, const float* norm_weight,
                                   int B, int H, int N, int d, int Dv, int causal,
                                   float lambda, float lambda_init, float eps, int in_dtype,
                                   const void* saved, size_t saved_bytes,
                                   float* dq1, float* dq2, float* dk1, float* dk2, float* dv,
                                   float* dlambda, float* dnorm_weight,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * diffattn_lambda_bwd — on the host, the gradients of
 *   lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init
 * with respect to the four vectors, given dlambda:
 *   dlq1 = dlambda e1 lk1, dlk1 = dlambda e1 lq1, dlq2 = -dlambda e2 lk2,
 *   dlk2 = -dlambda e2 lq2, with e1 = exp(lq1 . lk1), e2 = exp(lq2 . lk2)
 * (section "Como a atenção diferencial funciona"). Every pointer is a HOST
 * pointer to d floats; computed in double. INVALID_ARG on NULL pointers, d < 1
 * or a non-finite result.
 */
diffattn_status diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int d,
                                    float dlambda, float* dlq1, float* dlk1, float* dlq2, float* dlk2);

/*
 * diffattn_add_rmsnorm — the pre-RMSNorm and residual add of the DIFF
 * Transformer layer ("A Simple Principle From Noise-Cancelling Headphones...",
 * section "The Overall Architecture Of The Multi-Head Differential
 * Transformer": each block is pre-normalised with RMSNorm, as in LLaMA, and
 * added back to its input). Row by row: y = x + z (z optional) and
 * n = y / sqrt(mean(y^2) + eps) * weight (weight optional).
 *
 * x: [M, N] row-major contiguous, bf16 or f32 (x_dtype); z: [M, N] f32 or NULL.
 * y_out: [M, N] f32 or NULL (y is not written); n_out: [M, N] of n_dtype (bf16
 * or f16) or NULL.
 * weight: [N] f32 or NULL. N a multiple of 8; every pointer 16-byte aligned.
 * M equal to 0: returns DIFFATTN_OK.
 */
diffattn_status diffattn_add_rmsnorm(const void* x, int x_dtype, const float* z, float* y_out, void* n_out,
                                     int n_dtype, const float* weight, int M, int N, float eps, void* stream);

/*
 * diffattn_swiglu — the SwiGLU activation of the layer's feed-forward block
 * (same section: "Feed-forward network (FFN) (applying the SwiGLU activation
 * function)"; LLaMA's form): h = SiLU(g) * u, SiLU(t) = t / (1 + e^-t), where
 * each row of gate_up holds [g | u].
 *
 * gate_up: [M, 2H] f16 contiguous (the output of one GEMM against [W_gate |
 * W_up]); h_out: [M, H] contiguous, h_dtype bf16 or f16. H a multiple of 8;
 * pointers 16-byte aligned. M equal to 0: returns DIFFATTN_OK.
 */
diffattn_status diffattn_swiglu(const void* gate_up, void* h_out, int h_dtype, int M, int H, void* stream);

/*
 * diffattn_fwd_host — diffattn_fwd end to end from HOST buffers: the work is
 * split into pieces, each a range of heads of one batch entry (`chunks` asks for
 * that many pieces, 0 = 4, at most 16; every batch entry gets ceil(chunks / B)
 * head ranges); each piece's inputs are copied to the device, its prefill runs,
 * and its output is copied back, on three streams owned by the library, so that
 * the copies of one piece overlap the prefill and copies of others. One
 * cudaMemcpyAsync per input tensor piece (contiguous in [B, H, N, *]) and one
 * pitched cudaMemcpy2DAsync per output piece (a head range of [B, N, H, Dv]).
 * q1, q2, k1, k2: host [B, H, N, d] contiguous; v: host [B, H, N, Dv]
 * contiguous; out: host [B, N, H, Dv] contiguous; in_dtype / out_dtype, the
 * arguments from norm_weight (a DEVICE pointer or NULL) to eps, and the
 * supported shapes as for diffattn_fwd. Host buffers should be pinned (pageable
 * memory works, without overlap).
 * device_buffer: at least diffattn_fwd_host_buffer_size() bytes of device
 * memory, 256-byte aligned; its first 256 bytes are the workspace (the error
 * word, zero before the first call: diffattn_read_error(device_buffer, ...)),
 * the rest holds the device copies. Owned by the caller; one call at a time
 * per buffer.
 * Ordering: the call waits for work already enqueued on `stream` and makes
 * `stream` wait for its last copy back, so work enqueued on `stream` afterwards
 * (and a stream synchronisation) sees `out` filled. Concurrent calls from
 * several host threads are serialised (the library's streams are shared).
 * Errors: DIFFATTN_ERR_INVALID_ARG / _WORKSPACE before anything is enqueued;
 * those of diffattn_fwd; DIFFATTN_ERR_CUDA if a copy or stream call fails.
 */
diffattn_status diffattn_fwd_host(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                                  void* out, const float* norm_weight, int B, int H, int N, int d, int Dv, int causal,
                                  float lambda, float lambda_init, float eps, int in_dtype, int out_dtype, int chunks,
                                  void* device_buffer, size_t device_buffer_bytes, void* stream);
diffattn_status diffattn_fwd_host_buffer_size(int B, int H, int N, int d, int Dv, int in_dtype, int out_dtype,
                                              size_t* bytes);

/*
 * diffattn_gemm_bf16 — C[M, N] = A[M, K] . W[K, N], bf16 operands, fp32
 * accumulation, tcgen05 tensor cores. The module's projections: [Q|K|V] = X W
 * and Y = concat(heads) W_O ("A Simple Principle From Noise-Cancelling
 * Headphones...", sections "Moving On To The Differential Transformer" and
 * "Differential Attention With Multiple Heads").
 * A row-major with leading dimension lda (elements, K contiguous); W row-major
 * with ldw (N contiguous); C row-major with ldc, dtype out_dtype (f32, bf16 or
 * f16).
 * M, N, K >= 1; N a multiple of 8; pointers 16-byte aligned; lda, ldw
 * multiples of 8; ldc a multiple of 8 (bf16/f16 C) or 4 (f32 C). Ragged M, N and
 * K tiles are handled (out-of-range operand elements read as zero).
 * workspace: at least diffattn_gemm_workspace_size() bytes, 256-byte aligned
 *   (the error word, zero before the first call).
 */
diffattn_status diffattn_gemm_bf16(const void* A, const void* W, void* C, int M, int N, int K,
                                   int64_t lda, int64_t ldw, int64_t ldc, int out_dtype,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * diffattn_gemm_f16 — the same GEMM with fp16 operands A and W (arguments,
 * layout, alignment and errors as diffattn_gemm_bf16). fp16 keeps three more
 * mantissa bits than bf16 for operands of bounded range, such as the RMSNorm
 * outputs a DIFF Transformer layer multiplies.
 */
diffattn_status diffattn_gemm_f16(const void* A, const void* W, void* C, int M, int N, int K,
                                  int64_t lda, int64_t ldw, int64_t ldc, int out_dtype,
                                  void* workspace, size_t workspace_bytes, void* stream);

diffattn_status diffattn_gemm_workspace_size(int M, int N, int K, size_t* bytes);

/*
 * diffattn_gemm_residual — C = A . W + R in fp32 (tcgen05 GEMM with a fused
 * epilogue), for the DIFF Transformer layer's residual connections
 * Y = MultiHead(RMSNorm(X)) + X and X' = SwiGLU(RMSNorm(Y)) + Y ("The Overall
 * Architecture Of The Multi-Head Differential Transformer", intoai.pub;
 * "Estrutura multi-head e arquitetura completa", hada).
 * A [M, K] (lda) and W [K, N] (ldw) row-major, both ab_dtype (bf16 or f16);
 * R [M, N] row-major (ldr), r_dtype f32, bf16 or f16; C [M, N] fp32 (ldc).
 * Optional outputs (NULL to skip):
 *   C16 [M, N] (ldc16), c16_dtype bf16 or f16: C times c16_gain[N] (per column;
 *     NULL = 1), rounded — the next GEMM's operand, RMSNorm(C) W being
 *     (C (g W)) / r row by row;
 *   row_sq [M, N / 256] fp32: row m's sum of C^2 over columns 256 t .. 256 t + 255
 *     in entry m * (N / 256) + t (the partial sums of the RMSNorm's mean square).
 * N a multiple of 256; M, K >= 1; pointers 16-byte aligned (row_sq 4-byte);
 * lda, ldw, ldc16 multiples of 8, ldc a multiple of 4, ldr a multiple of 4
 * (fp32 R) or 8; c16_gain only with C16. Workspace as diffattn_gemm_bf16.
 * Errors: DIFFATTN_ERR_INVALID_ARG / _WORKSPACE before anything is launched.
 */
diffattn_status diffattn_gemm_residual(const void* A, const void* W, const void* R, float* C, void* C16,
                                       const float* c16_gain, float* row_sq, int M, int N, int K,
                                       int64_t lda, int64_t ldw, int64_t ldr, int64_t ldc, int64_t ldc16,
                                       int ab_dtype, int r_dtype, int c16_dtype,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * diffattn_gemm_swiglu — the feed-forward block's first product and SwiGLU in
 * one launch (same sections; "Feed-forward network (FFN) (applying the SwiGLU
 * activation function)"): H[m, j] = SiLU(g / r) * (u / r), SiLU(t) = t / (1 + e^-t),
 * where g and u are the gate and up columns of A . W_gu and r the RMS of row m of
 * the RMSNorm input: r = sqrt(sum_{t < n_sq} row_sq[m * n_sq + t] / sq_count + eps)
 * (r = 1 when row_sq is NULL). With A the unnormalised rows and the RMSNorm's gain
 * folded into A (diffattn_gemm_residual's c16_gain), this is SwiGLU(RMSNorm(.) W).
 * W_gu [K, 2F] row-major (ldw): gate and up blocks of 128 columns interleaved,
 * columns 256 t .. 256 t + 127 = W_gate columns 128 t .., 256 t + 128 .. 256 t + 255
 * = W_up columns 128 t ..; F a multiple of 128. A [M, K] (lda), ab_dtype bf16 or
 * f16 as W_gu; H [M, F] (ldh), h_dtype bf16 or f16. sq_count > 0 and eps >= 0
 * finite when row_sq is given, n_sq >= 1. Alignment, workspace and errors as
 * diffattn_gemm_bf16.
 */
diffattn_status diffattn_gemm_swiglu(const void* A, const void* W_gu, void* H, const float* row_sq, int n_sq,
                                     float sq_count, float eps, int M, int F, int K, int64_t lda, int64_t ldw,
                                     int64_t ldh, int ab_dtype, int h_dtype, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * diffattn_read_error — reads and clears the device error word at the start of
 * a workspace used by an earlier call. Synchronises `stream` (the one place the
 * library blocks). *device_code (host pointer) receives the raw code: 0 = none;
 * otherwise (site << 8) | kind, where kind 1 = a bounded wait gave up.
 * Returns DIFFATTN_ERR_TIMEOUT when the code is non-zero, DIFFATTN_OK when it
 * is zero, DIFFATTN_ERR_CUDA if the copy fails.
 */
diffattn_status diffattn_read_error(void* workspace, void* stream, int32_t* device_code);

/*
 * diffattn_selftest_timeout — exercises the bounded-wait path every kernel of
 * the library relies on: launches one CTA whose single barrier wait can never
 * complete. After about one second the wait gives up, records site 0x7F
 * (device code 0x7F01) in the workspace error word and the kernel returns; a
 * later diffattn_read_error on that workspace reports DIFFATTN_ERR_TIMEOUT.
 * workspace: at least 256 bytes, 256-byte aligned, error word zero.
 */
diffattn_status diffattn_selftest_timeout(void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H */
