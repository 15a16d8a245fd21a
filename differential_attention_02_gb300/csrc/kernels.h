// Internal launcher interface between the C-ABI layer (api.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace da {

// fp32 SIMT prefill (any d <= 128 multiple of 4, Dv <= 256 multiple of 32).
struct SimtF32Params {
    const float* q1;
    const float* q2;
    const float* k1;
    const float* k2;
    const float* v;
    int64_t sq1[3], sq2[3], sk1[3], sk2[3], sv[3];  // b, h, n strides in elements
    void* out;                                      // [B, N, H, Dv]
    int out_bf16;
    const float* norm_w;  // [Dv] or null
    int B, H, N, d, Dv, causal;
    float lambda, lambda_init, eps;
};
cudaError_t launch_fwd_simt_f32(const SimtF32Params& p, cudaStream_t stream);

// Backward pass on the CUDA cores (fp32 arithmetic; inputs fp32, bf16 or fp16).
struct BwdParams {
    const void *q1, *q2, *k1, *k2, *v;              // [B, H, N, d] / [B, H, N, Dv], in_dtype
    int64_t sq1[3], sq2[3], sk1[3], sk2[3], sv[3];  // b, h, n strides in elements
    const void* dy;                                 // [B, N, H, Dv] contiguous, in_dtype
    const float* norm_w;                            // [Dv] or null
    float *dq1, *dq2, *dk1, *dk2;                   // [B, H, N, d] contiguous
    float* dv;                                      // [B, H, N, Dv] contiguous
    float* dlambda;                                 // [1]
    float* dnorm_w;                                 // [Dv] or null
    float* d_o;                                     // workspace [B, H, N, Dv]
    float* stats;                                   // workspace [B, H, N, 4]: lse1, lse2, D1, D2
    float* part_lam;                                // workspace [partials]
    float* part_w;                                  // workspace [partials, Dv]
    int B, H, N, d, Dv, causal, in_dtype;           // in_dtype 0 fp32, 1 bf16, 2 fp16
    float lambda, lambda_init, eps;
};
int64_t bwd_partial_count(int B, int H, int N);
cudaError_t launch_bwd_simt(const BwdParams& p, cudaStream_t stream);
// Block 0: *dlambda = sum of n_part partials; block 1 + c: dnorm_w[c] (fixed order).
cudaError_t launch_bwd_reduce(const BwdParams& p, int64_t n_part, cudaStream_t stream);

// Backward on tcgen05 (d = 64, Dv = 128, bf16 or fp16 operands), after launch_bwd_prep.
struct BwdTcParams {
    CUtensorMap tm_q1, tm_q2, tm_k1, tm_k2, tm_v;  // 4-D maps over [B, H, N, width], boxes of 64 x 128 rows
    CUtensorMap tm_do;                             // dO [B, H, N, Dv], boxes of 64 x 128 rows
    CUtensorMap tm_q1s, tm_q2s, tm_dos;            // the same tensors in boxes of 64 x 64 rows (query steps)
    CUtensorMap tm_stats;                          // 2-D map over the stats [B*H*N][4] fp32, boxes of 4 x 64
    const float* stats;                            // [B, H, N, 4]: L1, L2, D1, D2
    float *dq1, *dq2, *dk1, *dk2, *dv;             // fp32 gradients, contiguous
    int B, H, N, d, Dv, causal, in_f16;
    float lambda, scale_log2, scale;               // scale = 1/sqrt(d), scale_log2 = log2(e)/sqrt(d)
    int32_t* err;
};
bool bwd_tc_supported(int d, int Dv, int in_dtype);  // in_dtype 1 bf16, 2 fp16
cudaError_t launch_bwd_tc(const BwdTcParams& p, cudaStream_t key_stream, cudaStream_t query_stream);  // key side, query side

// bf16 split-KV decode (+ merge).
struct DecodeParams {
    CUtensorMap tm_k1, tm_k2, tm_v;  // 4-D maps over [B, H_kv, L, width], or [pages, H_kv, 64, width] when paged
    const void* q1;                  // [B, H, d] bf16
    const void* q2;
    const int32_t* seq_lens;  // [B] or null
    int L;
    void* out;  // [B, H, Dv]
    int out_bf16;
    const float* norm_w;
    int B, H, d, Dv, num_splits, keys_per_split;
    float lambda, lambda_init, eps;
    float* part_stats;  // [B*H*S][4]
    float* part_o;      // [B*H*S][2][Dv]
    int32_t* err;
    const int32_t* block_table;  // [B][max_pages] physical page of each 64-token page, or null (contiguous cache)
    int max_pages;
    int num_pages = 0;           // pages in the pool (paged cache; checked in debug builds only)
    int kv_group;  // query heads per KV head (query head h reads KV head h / kv_group)
    int kv_fp8;    // cache of fp8 e4m3 values (1) or bf16 (0)
    float k1_scale = 1.f, k2_scale = 1.f, v_scale = 1.f;  // cache value = stored value * scale
};
cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream);
struct KvAppendParams {
    const void* k1_new;  // [B, H_kv, d] bf16, contiguous
    const void* k2_new;
    const void* v_new;   // [B, H_kv, Dv] bf16, contiguous
    void* k1_pages;      // [pages, H_kv, 64, d]: element strides below
    void* k2_pages;
    void* v_pages;
    int64_t k_stride_page, k_stride_h, k_stride_row;  // shared by k1_pages and k2_pages
    int64_t v_stride_page, v_stride_h, v_stride_row;
    const int32_t* block_table;  // [B][max_pages]
    const int32_t* seq_lens;     // [B]: the new token is at position seq_lens[b] - 1
    int max_pages, num_pages, B, H_kv, d, Dv;
    int fp8;                                          // pages hold fp8 e4m3: store sat(x / scale)
    float k1_scale = 1.f, k2_scale = 1.f, v_scale = 1.f;
};
cudaError_t launch_kv_append_paged(const KvAppendParams& p, cudaStream_t stream);

struct AddNormParams {
    const void* x;        // [M, N] bf16 or fp32 (x_f32)
    int x_f32;
    const float* z;       // [M, N] fp32 added to x, or null
    float* y_out;         // [M, N] fp32 = x + z, or null
    void* n_out;          // [M, N] bf16 or fp16 (n_f16) = RMSNorm(x + z) * weight, or null
    int n_f16;
    const float* weight;  // [N] or null
    int M, N;
    float eps;
};
cudaError_t launch_add_rmsnorm(const AddNormParams& p, cudaStream_t stream);
cudaError_t launch_swiglu(const void* gate_up, void* h, int h_f16, int64_t M, int H, cudaStream_t stream);
int decode_keys_per_stage(int d);

// bf16 GEMM on tcgen05: C = A * W.
struct GemmParams {
    CUtensorMap tm_a;  // [M, K] K-major, box {64, 128}, 128B swizzle
    CUtensorMap tm_w;  // [K, N] N-major, box {64, 64}, 128B swizzle
    CUtensorMap tm_c;  // [M, N] output, boxes of 128 bytes x 32 rows, 128B swizzle
    void* C;
    int64_t ldc;
    int M, N, K, out_bf16, out_f16;  // output bf16, fp16, or fp32 when both are 0
    int ab_f16;                      // operands A and W fp16 (1) or bf16 (0)
    int32_t* err;
    // Epilogue. mode 0: C = A.W. mode 1 (residual): C = A.W + R in fp32 (N a multiple of
    // 256); optionally a 16-bit copy C * gain and per-tile row sums of C^2. mode 2
    // (SwiGLU): the columns of W are gate and up blocks of 128 interleaved per 256-column
    // tile; C[m, j] = silu(g / r) * (u / r), C has N / 2 columns, r the row's RMS from
    // the partial sums of squares row_sq_in (r = 1 without them).
    int mode = 0;
    const void* resid = nullptr;     // mode 1: R [M, N], row stride ld_r elements
    int64_t ld_r = 0;
    int r_dtype = 0;                 // 0 fp32, 1 bf16, 2 fp16
    void* c16 = nullptr;             // mode 1 (optional): 16-bit copy, row stride ld_c16 elements
    int64_t ld_c16 = 0;
    int c16_f16 = 0;                 // copy fp16 (1) or bf16 (0)
    const float* c16_gain = nullptr; // mode 1 (optional): per-column factor of the copy
    float* row_sq = nullptr;         // mode 1 (optional): [M, N / 256] sums of C^2 per 256-column tile
    const float* row_sq_in = nullptr;  // mode 2 (optional): [M, n_sq] partial sums of squares
    int n_sq = 0;
    float sq_count = 1.f, eps = 0.f; // mode 2: r = sqrt(sum / sq_count + eps)
};
cudaError_t launch_gemm_bf16(const GemmParams& p, cudaStream_t stream);
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;

// bf16 fused prefill on tcgen05.
struct FwdParams {
    CUtensorMap tm_q1, tm_q2, tm_k1, tm_k2, tm_v;  // 4-D maps over [B, H, N, width]
    CUtensorMap tm_out;                            // 3-D map over the output [B, N, H*Dv], 128-byte boxes
    CUtensorMap tm_dy;                             // backward preparation: dy [B, N, H*Dv], boxes as tm_out
    void* out;                                     // [B, N, H, Dv]
    int out_bf16, out_f16;                         // output bf16, fp16, or fp32 when both are 0
    int in_f16;                                    // operands fp16 (1) or bf16 (0)
    const float* norm_w;
    int B, H, N, d, Dv, causal;
    float lambda, lambda_init, eps;
    float scale_log2;  // log2(e) / sqrt(d)
    int32_t* err;
    // Backward preparation (launch_bwd_prep): the same forward, whose epilogue
    // writes what the tensor-core backward needs instead of the output.
    const void* dy = nullptr;      // [B, N, H, Dv] output gradient, operand dtype
    void* d_o = nullptr;           // [B, H, N, Dv] gradient of the pre-norm output, operand dtype
    float* stats = nullptr;        // [B, H, N, 4]: log2 sum-exp of map 1, of map 2 (scaled-score units), D1, D2
    float* part_lam = nullptr;     // [grid] per-CTA partial of dlambda
    float* part_w = nullptr;       // [grid][Dv] per-CTA partial of the gain's gradient
    // Training forward (launch_fwd_train) writes, besides the output, the state the
    // backward starts from; launch_bwd_prep_saved reads it instead of re-running the forward.
    float* x_save = nullptr;       // [B, H, N, Dv]: x = O1/l1 - lambda O2/l2, the output before the norm (fp32)
    void* a2_save = nullptr;       // [B, H, N, Dv]: O2/l2, map 2's own output, in the operand type
    CUtensorMap tm_xsave;          // 3-D map over x_save [B H][N][Dv] fp32, boxes of 32 x 128 rows
    CUtensorMap tm_a2save;         // 3-D map over a2_save [B H][N][Dv] 16-bit, boxes of 64 x 128 rows
    float* lse_save = nullptr;     // [B, H, N, 2]: L1, L2 = max + log2(sum) per map (base 2, scaled scores)
};
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream);       // both maps in one CTA
cudaError_t launch_fwd_train(const FwdParams& p, cudaStream_t stream);      // d=64: forward + saved state
cudaError_t launch_bwd_prep(const FwdParams& p, cudaStream_t stream);       // d=64: forward + backward inputs
cudaError_t launch_bwd_prep_saved(const FwdParams& p, cudaStream_t stream); // d=64: backward inputs from the saved state
cudaError_t launch_fwd_pair_bf16(const FwdParams& p, cudaStream_t stream);  // one map per CTA of a pair
constexpr int kFwdBM = 128;
constexpr int kFwdBN = 128;

// One CTA whose single wait can never complete (bounded-wait self-test).
cudaError_t launch_selftest_timeout(int32_t* err, cudaStream_t stream);

// One-time setup of a kernel on the current device (first call per device):
// the dynamic shared-memory opt-in and, when want_regs > 0, a check that the
// compiled per-thread register count is the one the kernel's register split
// was computed from. Later calls on that device return at once.
template <auto Kernel>
cudaError_t prepare_once(int smem_bytes, int want_regs = 0) {
    static std::atomic<uint64_t> ready{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit != 0 && (ready.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    if (want_regs > 0) {
        cudaFuncAttributes a;
        e = cudaFuncGetAttributes(&a, Kernel);
        if (e != cudaSuccess) return e;
        if (a.numRegs != want_regs) return cudaErrorInvalidConfiguration;
    }
    ready.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
}

// Launches `kernel` as a programmatic dependent of the previous kernel in `stream`: its CTAs
// may start (and run their setup up to pdl_wait) while that kernel's last CTAs finish.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Number of SMs of the current device (queried once per device).
inline cudaError_t device_sm_count(int* sms) {
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && (*sms = cache[dev].load(std::memory_order_relaxed)) > 0) return cudaSuccess;
    if ((e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev < 64) cache[dev].store(*sms, std::memory_order_relaxed);
    return cudaSuccess;
}

}  // namespace da
