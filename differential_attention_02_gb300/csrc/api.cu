// Host side of the C ABI declared in include/diffattn.h: argument checks,
// TMA descriptor encoding, kernel dispatch. No device memory is allocated
// here and nothing synchronises except diffattn_read_error.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/diffattn.h"
#include "common.cuh"
#include "kernels.h"

using namespace da;

namespace {
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// ---------------------------------------------------------------- helpers
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

int device_sm_count() {
    int n = 0;
    return da::device_sm_count(&n) == cudaSuccess ? n : 0;
}

// 4-D bf16 map over a [B, H, rows, width] operand (strides in elements).
// Size-1 dimensions get a harmless stride, since their stride is never used.
bool encode_4d(CUtensorMap* m, const diffattn_tensor& t, int width, int rows, int H, int B, int box_w, int box_rows,
               CUtensorMapSwizzle sw, CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int eb = dt == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1 : 2;  // bytes per element
    const int64_t sn = t.stride_n, sh = (H > 1) ? t.stride_h : (int64_t)rows * sn,
                  sb = (B > 1) ? t.stride_b : (int64_t)H * sh;
    cuuint64_t dims[4] = {(cuuint64_t)width, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(sn * eb), (cuuint64_t)(sh * eb), (cuuint64_t)(sb * eb)};
    cuuint32_t box[4] = {(cuuint32_t)box_w, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void*>(t.ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a contiguous output [B, N, W] (W = H * Dv elements per token),
// boxes of 128 bytes x `box_rows` rows, 128-byte swizzle (for TMA stores).
bool encode_out_3d(CUtensorMap* m, void* ptr, int W, int N, int B, int elem_bytes, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)N, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)W * elem_bytes, (cuuint64_t)W * elem_bytes * N};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the backward's per-row statistics [rows][4] fp32, boxes of 4 x 64
// rows, unswizzled (the key-side gradient kernel loads one query step at a time).
bool encode_stats_2d(CUtensorMap* m, const float* ptr, int64_t rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {4, (cuuint64_t)rows};
    cuuint64_t strides[1] = {16};
    cuuint32_t box[2] = {4, 64};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d(CUtensorMap* m, const void* ptr, int inner, int outer, int64_t ld, int box_inner, int box_outer,
               bool f16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    cuuint32_t es[2] = {1, 1};
    return enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr),
               dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand [B, H, rows, width], last dim contiguous; strides in elements; every
// byte stride a multiple of 16 and the row stride at least the width.
bool check_operand(const diffattn_tensor& t, int width, int elem_bytes) {
    if (t.ptr == nullptr || !aligned16(t.ptr)) return false;
    const int64_t q = 16 / elem_bytes;
    if (t.stride_n < width || t.stride_n % q) return false;
    if (t.stride_h < 0 || t.stride_h % q || t.stride_b < 0 || t.stride_b % q) return false;
    return true;
}

diffattn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DIFFATTN_OK : DIFFATTN_ERR_CUDA; }

int32_t* err_word(void* ws) { return reinterpret_cast<int32_t*>(ws); }

// Decode split count: the smallest split count whose CTA waves are at least 90%
// full on this GPU, capped so that every split keeps at least 256 keys.
int decode_auto_splits(int B, int H, int L, int d, bool fp8) {
    const int n_sm = device_sm_count();
    const int sms = n_sm > 0 ? n_sm : 148;
    // Resident split CTAs per SM (bound by shared memory; fp8 stages are half the bytes).
    const int per_sm = (d == 64) ? (fp8 ? 3 : 2) : 1;
    const double slots = (double)sms * per_sm;
    const int smax = std::max(1, std::min(256, L / 256));
    for (int s = 1; s <= smax; ++s) {
        const double waves = (double)B * H * s / slots;
        if (waves >= 1.0 && waves / ceil(waves) >= 0.9) return s;
        if (waves < 1.0 && s == smax) return s;
    }
    return smax;
}

void decode_geometry(int B, int H, int L, int d, int num_splits, int* S, int* kps, bool fp8 = false) {
    int s = num_splits > 0 ? num_splits : decode_auto_splits(B, H, L, d, fp8);
    const int stage = decode_keys_per_stage(d);
    int k = (L + s - 1) / s;
    k = (k + stage - 1) / stage * stage;
    s = (L + k - 1) / k;  // no split left without keys
    *S = s;
    *kps = k;
}

size_t decode_ws_bytes(int B, int H, int S, int Dv) {
    return kControlBytes + (size_t)B * H * S * 4 * sizeof(float) + (size_t)B * H * S * 2 * Dv * sizeof(float);
}

}  // namespace

extern "C" {

const char* diffattn_status_string(int s) {
    switch (s) {
        case DIFFATTN_OK: return "ok";
        case DIFFATTN_ERR_INVALID_ARG: return "invalid argument";
        case DIFFATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case DIFFATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case DIFFATTN_ERR_CUDA: return "CUDA error";
        case DIFFATTN_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

diffattn_status diffattn_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int d,
                                int layer, float lambda_init_override, float* lambda_out, float* lambda_init_out) {
    if (!lq1 || !lk1 || !lq2 || !lk2 || !lambda_out || !lambda_init_out || d < 1) return DIFFATTN_ERR_INVALID_ARG;
    double lam_init;
    if (lambda_init_override >= 0.f) {
        lam_init = lambda_init_override;
    } else {
        if (layer < 1) return DIFFATTN_ERR_INVALID_ARG;
        lam_init = 0.8 - 0.6 * exp(-0.3 * (double)(layer - 1));
    }
    double d1 = 0.0, d2 = 0.0;
    for (int i = 0; i < d; ++i) {
        d1 += (double)lq1[i] * (double)lk1[i];
        d2 += (double)lq2[i] * (double)lk2[i];
    }
    const double lam = exp(d1) - exp(d2) + lam_init;
    if (!isfinite(lam)) return DIFFATTN_ERR_INVALID_ARG;
    *lambda_out = (float)lam;
    *lambda_init_out = (float)lam_init;
    return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_workspace_size(int B, int H, int N, int d, int Dv, size_t* bytes) {
    if (!bytes || B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    *bytes = kControlBytes;
    return DIFFATTN_OK;
}

}  // extern "C"

namespace {
struct SavedLayout {
    size_t x, a2, lse, total;  // x (fp32), O2/l2 (16-bit), L1 and L2 per row (fp32)
};
SavedLayout saved_layout(int B, int H, int N, int Dv) {
    const size_t rows = (size_t)B * H * N;
    SavedLayout l;
    l.x = 0;
    l.a2 = round256(rows * Dv * sizeof(float));
    l.lse = l.a2 + round256(rows * Dv * sizeof(uint16_t));
    l.total = l.lse + round256(rows * 2 * sizeof(float));
    return l;
}
bool saved_ok(const void* saved, size_t bytes, int B, int H, int N, int Dv) {
    return saved != nullptr && !(reinterpret_cast<uintptr_t>(saved) & 255u) && bytes >= saved_layout(B, H, N, Dv).total;
}

// diffattn_fwd, and with `saved` set the training forward (tensor-core path,
// d=64/Dv=128; the caller has checked that).
diffattn_status fwd_impl(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                         diffattn_tensor v, void* out, const float* norm_weight, int B, int H, int N, int d, int Dv,
                         int causal, float lambda, float lambda_init, float eps, int in_dtype, int out_dtype,
                         void* workspace, size_t workspace_bytes, void* stream, void* saved) {
    if (B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if ((in_dtype != DIFFATTN_F32 && in_dtype != DIFFATTN_BF16 && in_dtype != DIFFATTN_F16) ||
        (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16 && out_dtype != DIFFATTN_F16) ||
        (in_dtype == DIFFATTN_F32 && out_dtype == DIFFATTN_F16))
        return DIFFATTN_ERR_INVALID_ARG;
    if (!isfinite(lambda) || !isfinite(lambda_init) || !(eps >= 0.f) || !isfinite(eps))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || N == 0) return DIFFATTN_OK;
    const int eb = in_dtype == DIFFATTN_F32 ? 4 : 2;
    if (!check_operand(q1, d, eb) || !check_operand(q2, d, eb) || !check_operand(k1, d, eb) ||
        !check_operand(k2, d, eb) || !check_operand(v, Dv, eb))
        return DIFFATTN_ERR_INVALID_ARG;
    if (out == nullptr || !aligned16(out)) return DIFFATTN_ERR_INVALID_ARG;
    if (norm_weight != nullptr && !aligned16(norm_weight)) return DIFFATTN_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < kControlBytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (in_dtype == DIFFATTN_F32) {
        if (d > 128 || d % 4 || Dv > 256 || Dv % 32) return DIFFATTN_ERR_UNSUPPORTED;
        SimtF32Params p{};
        p.q1 = static_cast<const float*>(q1.ptr);
        p.q2 = static_cast<const float*>(q2.ptr);
        p.k1 = static_cast<const float*>(k1.ptr);
        p.k2 = static_cast<const float*>(k2.ptr);
        p.v = static_cast<const float*>(v.ptr);
        const diffattn_tensor* ts[5] = {&q1, &q2, &k1, &k2, &v};
        int64_t* ss[5] = {p.sq1, p.sq2, p.sk1, p.sk2, p.sv};
        for (int i = 0; i < 5; ++i) {
            ss[i][0] = ts[i]->stride_b;
            ss[i][1] = ts[i]->stride_h;
            ss[i][2] = ts[i]->stride_n;
        }
        p.out = out;
        p.out_bf16 = out_dtype == DIFFATTN_BF16;
        p.norm_w = norm_weight;
        p.B = B; p.H = H; p.N = N; p.d = d; p.Dv = Dv; p.causal = causal != 0;
        p.lambda = lambda; p.lambda_init = lambda_init; p.eps = eps;
        return cuda_status(launch_fwd_simt_f32(p, st));
    }

    if (!((d == 64 && Dv == 128) || (d == 128 && Dv == 256))) return DIFFATTN_ERR_UNSUPPORTED;
    FwdParams p{};
    const CUtensorMapDataType dt =
        in_dtype == DIFFATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!encode_4d(&p.tm_q1, q1, d, N, H, B, 64, kFwdBM, sw, dt) || !encode_4d(&p.tm_q2, q2, d, N, H, B, 64, kFwdBM, sw, dt) ||
        !encode_4d(&p.tm_k1, k1, d, N, H, B, 64, kFwdBN, sw, dt) || !encode_4d(&p.tm_k2, k2, d, N, H, B, 64, kFwdBN, sw, dt) ||
        // V boxes: 128 keys for the single-CTA kernel, 64 for the CTA pair (half-tile V ring).
        !encode_4d(&p.tm_v, v, Dv, N, H, B, 64, d == 64 ? kFwdBN : kFwdBN / 2, sw, dt) ||
        !encode_out_3d(&p.tm_out, out, H * Dv, N, B, out_dtype == DIFFATTN_F32 ? 4 : 2, kFwdBM))
        return DIFFATTN_ERR_INVALID_ARG;
    p.in_f16 = in_dtype == DIFFATTN_F16;
    p.out = out;
    p.out_bf16 = out_dtype == DIFFATTN_BF16;
    p.out_f16 = out_dtype == DIFFATTN_F16;
    p.norm_w = norm_weight;
    p.B = B; p.H = H; p.N = N; p.d = d; p.Dv = Dv; p.causal = causal != 0;
    p.lambda = lambda; p.lambda_init = lambda_init; p.eps = eps;
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
    p.err = err_word(workspace);
    if (saved != nullptr) {
        const SavedLayout sl = saved_layout(B, H, N, Dv);
        uint8_t* sv = static_cast<uint8_t*>(saved);
        p.x_save = reinterpret_cast<float*>(sv + sl.x);
        p.a2_save = sv + sl.a2;
        p.lse_save = reinterpret_cast<float*>(sv + sl.lse);
        if (!encode_out_3d(&p.tm_xsave, p.x_save, Dv, N, B * H, 4, kFwdBM) ||
            !encode_out_3d(&p.tm_a2save, p.a2_save, Dv, N, B * H, 2, kFwdBM))
            return DIFFATTN_ERR_INVALID_ARG;
        return cuda_status(launch_fwd_train(p, st));
    }
    // (64, 128): both maps share one CTA; (128, 256): the accumulators of both
    // maps do not fit one CTA's tensor memory, so a CTA pair splits the maps.
    return cuda_status(d == 64 ? launch_fwd_bf16(p, st) : launch_fwd_pair_bf16(p, st));
}

// The training forward's saved state: O1, O2 (fp32 [2][B, H, N, Dv]), then the
// per-row max and sum of both maps (fp32 [B, H, N, 4]), each part 256-byte aligned.
}  // namespace

extern "C" {

diffattn_status diffattn_fwd(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                             diffattn_tensor v, void* out, const float* norm_weight, int B, int H, int N, int d,
                             int Dv, int causal, float lambda, float lambda_init, float eps, int in_dtype,
                             int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(q1, q2, k1, k2, v, out, norm_weight, B, H, N, d, Dv, causal, lambda, lambda_init, eps, in_dtype,
                    out_dtype, workspace, workspace_bytes, stream, nullptr);
}

diffattn_status diffattn_train_saved_size(int B, int H, int N, int Dv, size_t* bytes) {
    if (!bytes || B < 0 || H < 0 || N < 0 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    *bytes = saved_layout(B, H, N, Dv).total;
    return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_train(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                                   diffattn_tensor v, void* out, const float* norm_weight, int B, int H, int N, int d,
                                   int Dv, int causal, float lambda, float lambda_init, float eps, int in_dtype,
                                   int out_dtype, void* saved, size_t saved_bytes, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    if (in_dtype == DIFFATTN_F32) return DIFFATTN_ERR_UNSUPPORTED;
    if (B > 0 && H > 0 && N > 0 && !(d == 64 && Dv == 128)) return DIFFATTN_ERR_UNSUPPORTED;
    if (B > 0 && H > 0 && N > 0 && !saved_ok(saved, saved_bytes, B, H, N, Dv)) return DIFFATTN_ERR_INVALID_ARG;
    return fwd_impl(q1, q2, k1, k2, v, out, norm_weight, B, H, N, d, Dv, causal, lambda, lambda_init, eps, in_dtype,
                    out_dtype, workspace, workspace_bytes, stream, saved);
}

diffattn_status diffattn_decode_workspace_size(int B, int H, int L, int d, int Dv, int num_splits, size_t* bytes) {
    if (!bytes || B < 0 || H < 0 || L < 1 || d < 1 || Dv < 1 || num_splits < 0 || num_splits > 256)
        return DIFFATTN_ERR_INVALID_ARG;
    // Enough for either cache type: the fp8 decode may choose more splits.
    int S, S8, kps;
    decode_geometry(B, H, L, d, num_splits, &S, &kps, false);
    decode_geometry(B, H, L, d, num_splits, &S8, &kps, true);
    *bytes = decode_ws_bytes(B, H, std::max(S, S8), Dv);
    return DIFFATTN_OK;
}

}  // extern "C"

namespace {
// Every host check of diffattn_decode except the workspace: sizes, dtypes,
// scalars, pointers, alignment, operand strides and the (d, Dv) pair. With
// B == 0 or H == 0 only the size, dtype and scalar checks apply (nothing runs).
diffattn_status decode_check_args(const void* q1, const void* q2, const diffattn_tensor& k1_cache,
                                  const diffattn_tensor& k2_cache, const diffattn_tensor& v_cache, int L,
                                  const void* out, const float* norm_weight, int B, int H, int d, int Dv, float lambda,
                                  float lambda_init, float eps, int num_splits, int out_dtype) {
    if (B < 0 || H < 0 || L < 1 || d < 1 || Dv < 1 || num_splits < 0 || num_splits > 256)
        return DIFFATTN_ERR_INVALID_ARG;
    if (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if (!isfinite(lambda) || !isfinite(lambda_init) || !(eps >= 0.f) || !isfinite(eps))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return DIFFATTN_OK;
    if (!q1 || !q2 || !aligned16(q1) || !aligned16(q2) || !out || !aligned16(out)) return DIFFATTN_ERR_INVALID_ARG;
    if (!check_operand(k1_cache, d, 2) || !check_operand(k2_cache, d, 2) || !check_operand(v_cache, Dv, 2))
        return DIFFATTN_ERR_INVALID_ARG;
    if (norm_weight != nullptr && !aligned16(norm_weight)) return DIFFATTN_ERR_INVALID_ARG;
    if (!((d == 64 && Dv == 128) || (d == 128 && Dv == 256))) return DIFFATTN_ERR_UNSUPPORTED;
    return DIFFATTN_OK;
}
}  // namespace

extern "C" {

diffattn_status diffattn_decode(const void* q1, const void* q2, diffattn_tensor k1_cache, diffattn_tensor k2_cache,
                                diffattn_tensor v_cache, const int32_t* seq_lens, int L, void* out,
                                const float* norm_weight, int B, int H, int d, int Dv, float lambda,
                                float lambda_init, float eps, int num_splits, int out_dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
    const diffattn_status chk = decode_check_args(q1, q2, k1_cache, k2_cache, v_cache, L, out, norm_weight, B, H, d,
                                                  Dv, lambda, lambda_init, eps, num_splits, out_dtype);
    if (chk != DIFFATTN_OK || B == 0 || H == 0) return chk;
    DecodeParams p{};
    decode_geometry(B, H, L, d, num_splits, &p.num_splits, &p.keys_per_split);
    const size_t need = decode_ws_bytes(B, H, p.num_splits, Dv);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    const int stage = decode_keys_per_stage(d);
    if (!encode_4d(&p.tm_k1, k1_cache, d, L, H, B, 64, stage, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_4d(&p.tm_k2, k2_cache, d, L, H, B, 64, stage, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_4d(&p.tm_v, v_cache, Dv, L, H, B, Dv, stage, CU_TENSOR_MAP_SWIZZLE_NONE))
        return DIFFATTN_ERR_INVALID_ARG;
    p.q1 = q1;
    p.q2 = q2;
    p.seq_lens = seq_lens;
    p.L = L;
    p.out = out;
    p.out_bf16 = out_dtype == DIFFATTN_BF16;
    p.norm_w = norm_weight;
    p.B = B; p.H = H; p.d = d; p.Dv = Dv;
    p.lambda = lambda; p.lambda_init = lambda_init; p.eps = eps;
    p.kv_group = 1;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.err = err_word(workspace);
    p.part_stats = reinterpret_cast<float*>(ws + kControlBytes);
    p.part_o = p.part_stats + (size_t)B * H * p.num_splits * 4;
    return cuda_status(launch_decode_bf16(p, static_cast<cudaStream_t>(stream)));
}

namespace {

// Byte offsets of the backward's workspace regions after the control block.
struct BwdLayout {
    size_t d_o, stats, part_lam, part_w, total;
};
BwdLayout bwd_layout(int B, int H, int N, int Dv) {
    const size_t rows = (size_t)B * H * N;
    const size_t parts = (size_t)bwd_partial_count(B, H, N);
    BwdLayout l;
    l.d_o = kControlBytes;
    l.stats = l.d_o + round256(rows * Dv * sizeof(float));
    l.part_lam = l.stats + round256(rows * 4 * sizeof(float));
    l.part_w = l.part_lam + round256(parts * sizeof(float));
    l.total = l.part_w + round256(parts * Dv * sizeof(float));
    return l;
}
}  // namespace

diffattn_status diffattn_bwd_workspace_size(int B, int H, int N, int d, int Dv, size_t* bytes) {
    if (!bytes || B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    *bytes = bwd_layout(B, H, N, Dv).total;
    return DIFFATTN_OK;
}

}  // extern "C"

namespace {
// diffattn_bwd, and with `saved` set the backward from a training forward's saved
// state (tensor-core path only; the caller has checked the saved buffer).
// One non-blocking side stream and a fork/join event pair per device, made on first
// use and kept for the life of the process. The mutex orders concurrent callers'
// fork, launches and join on the shared stream.
struct SideStream {
    std::mutex mu;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream() {
    static std::mutex init_mu;
    static SideStream sides[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(init_mu);
    SideStream& s = sides[dev];
    if (s.stream == nullptr) {
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    }
    return &s;
}

diffattn_status bwd_impl(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                         diffattn_tensor v, const void* dy, const float* norm_weight, int B, int H, int N, int d, int Dv,
                         int causal, float lambda, float lambda_init, float eps, int in_dtype, float* dq1, float* dq2,
                         float* dk1, float* dk2, float* dv, float* dlambda, float* dnorm_weight, void* workspace,
                         size_t workspace_bytes, void* stream, const void* saved) {
    if (B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (in_dtype != DIFFATTN_F32 && in_dtype != DIFFATTN_BF16 && in_dtype != DIFFATTN_F16)
        return DIFFATTN_ERR_INVALID_ARG;
    if (!isfinite(lambda) || !isfinite(lambda_init) || !(eps >= 0.f) || !isfinite(eps))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || N == 0) return DIFFATTN_OK;
    const int eb = in_dtype == DIFFATTN_F32 ? 4 : 2;
    if (!check_operand(q1, d, eb) || !check_operand(q2, d, eb) || !check_operand(k1, d, eb) ||
        !check_operand(k2, d, eb) || !check_operand(v, Dv, eb))
        return DIFFATTN_ERR_INVALID_ARG;
    const void* outs[8] = {dy, dq1, dq2, dk1, dk2, dv, dlambda, nullptr};
    for (int i = 0; i < 7; ++i)
        if (!outs[i] || !aligned16(outs[i])) return DIFFATTN_ERR_INVALID_ARG;
    if ((norm_weight && !aligned16(norm_weight)) || (dnorm_weight && !aligned16(dnorm_weight)))
        return DIFFATTN_ERR_INVALID_ARG;
    if (d % 32 || d > 128 || Dv % 32 || Dv > 256) return DIFFATTN_ERR_UNSUPPORTED;
    const BwdLayout lay = bwd_layout(B, H, N, Dv);
    if (workspace == nullptr || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    BwdParams p{};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.dlambda = dlambda;
    p.dnorm_w = dnorm_weight;
    p.Dv = Dv;
    p.part_lam = reinterpret_cast<float*>(ws + lay.part_lam);
    p.part_w = reinterpret_cast<float*>(ws + lay.part_w);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int dt = in_dtype == DIFFATTN_F32 ? 0 : in_dtype == DIFFATTN_BF16 ? 1 : 2;
    if (saved != nullptr && !bwd_tc_supported(d, Dv, dt)) return DIFFATTN_ERR_UNSUPPORTED;
    if (bwd_tc_supported(d, Dv, dt)) {
        // Tensor-core path: the forward re-run with the preparation epilogue (dO in
        // the operand type, per-row statistics, dlambda and gain partials), the
        // key-side and query-side gradient kernels, then the fixed-order reduction.
        const CUtensorMapDataType tdt = dt == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
        void* d_o = ws + lay.d_o;
        float* stats = reinterpret_cast<float*>(ws + lay.stats);
        const diffattn_tensor dot{d_o, (int64_t)H * N * Dv, (int64_t)N * Dv, Dv};
        FwdParams f{};
        if (!encode_4d(&f.tm_q1, q1, d, N, H, B, 64, kFwdBM, sw, tdt) ||
            !encode_4d(&f.tm_q2, q2, d, N, H, B, 64, kFwdBM, sw, tdt) ||
            !encode_4d(&f.tm_k1, k1, d, N, H, B, 64, kFwdBN, sw, tdt) ||
            !encode_4d(&f.tm_k2, k2, d, N, H, B, 64, kFwdBN, sw, tdt) ||
            !encode_4d(&f.tm_v, v, Dv, N, H, B, 64, kFwdBN, sw, tdt) ||
            !encode_out_3d(&f.tm_dy, const_cast<void*>(dy), H * Dv, N, B, 2, kFwdBM))
            return DIFFATTN_ERR_INVALID_ARG;
        f.in_f16 = dt == 2;
        f.norm_w = norm_weight;
        f.B = B; f.H = H; f.N = N; f.d = d; f.Dv = Dv; f.causal = causal != 0;
        f.lambda = lambda; f.lambda_init = lambda_init; f.eps = eps;
        f.scale_log2 = (float)(1.4426950408889634 / sqrt((double)d));
        f.err = err_word(workspace);
        f.dy = dy;
        f.d_o = d_o;
        f.stats = stats;
        f.part_lam = p.part_lam;
        f.part_w = p.part_w;
        BwdTcParams t{};
        t.tm_q1 = f.tm_q1; t.tm_q2 = f.tm_q2; t.tm_k1 = f.tm_k1; t.tm_k2 = f.tm_k2; t.tm_v = f.tm_v;
        if (!encode_4d(&t.tm_do, dot, Dv, N, H, B, 64, 128, sw, tdt) ||
            !encode_4d(&t.tm_q1s, q1, d, N, H, B, 64, 64, sw, tdt) ||
            !encode_4d(&t.tm_q2s, q2, d, N, H, B, 64, 64, sw, tdt) ||
            !encode_4d(&t.tm_dos, dot, Dv, N, H, B, 64, 64, sw, tdt) ||
            !encode_stats_2d(&t.tm_stats, stats, (int64_t)B * H * N))
            return DIFFATTN_ERR_INVALID_ARG;
        t.stats = stats;
        t.dq1 = dq1; t.dq2 = dq2; t.dk1 = dk1; t.dk2 = dk2; t.dv = dv;
        t.B = B; t.H = H; t.N = N; t.d = d; t.Dv = Dv; t.causal = causal != 0; t.in_f16 = dt == 2;
        t.lambda = lambda;
        t.scale_log2 = f.scale_log2;
        t.scale = (float)(1.0 / sqrt((double)d));
        t.err = err_word(workspace);
        cudaError_t e;
        if (saved != nullptr) {
            // The forward's state was saved: only the per-row preparation remains.
            const SavedLayout sl = saved_layout(B, H, N, Dv);
            uint8_t* sv = static_cast<uint8_t*>(const_cast<void*>(saved));
            f.x_save = reinterpret_cast<float*>(sv + sl.x);
            f.a2_save = sv + sl.a2;
            f.lse_save = reinterpret_cast<float*>(sv + sl.lse);
            e = launch_bwd_prep_saved(f, st);
        } else {
            e = launch_bwd_prep(f, st);
        }
        if (e != cudaSuccess) return cuda_status(e);
        // The key-side kernel stays on the caller's stream; the query-side kernel and
        // the reduction (both need only the preparation) go to a side stream forked
        // after the preparation and joined back before return, so their tails overlap.
        SideStream* side = side_stream();
        if (side == nullptr) return DIFFATTN_ERR_CUDA;
        std::lock_guard<std::mutex> lock(side->mu);
        if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess)
            return cuda_status(e);
        e = launch_bwd_tc(t, st, side->stream);
        if (e == cudaSuccess) e = launch_bwd_reduce(p, (int64_t)((N + kFwdBM - 1) / kFwdBM) * B * H, side->stream);
        const cudaError_t rj = cudaEventRecord(side->join, side->stream);
        const cudaError_t wj = cudaStreamWaitEvent(st, side->join, 0);
        if (e == cudaSuccess) e = rj != cudaSuccess ? rj : wj;
        return cuda_status(e);
    }
    p.q1 = q1.ptr; p.q2 = q2.ptr; p.k1 = k1.ptr; p.k2 = k2.ptr; p.v = v.ptr;
    const diffattn_tensor* ts[5] = {&q1, &q2, &k1, &k2, &v};
    int64_t* ss[5] = {p.sq1, p.sq2, p.sk1, p.sk2, p.sv};
    for (int i = 0; i < 5; ++i) {
        ss[i][0] = ts[i]->stride_b;
        ss[i][1] = ts[i]->stride_h;
        ss[i][2] = ts[i]->stride_n;
    }
    p.dy = dy;
    p.norm_w = norm_weight;
    p.dq1 = dq1; p.dq2 = dq2; p.dk1 = dk1; p.dk2 = dk2; p.dv = dv;
    p.d_o = reinterpret_cast<float*>(ws + lay.d_o);
    p.stats = reinterpret_cast<float*>(ws + lay.stats);
    p.B = B; p.H = H; p.N = N; p.d = d; p.causal = causal != 0;
    p.in_dtype = dt;
    p.lambda = lambda; p.lambda_init = lambda_init; p.eps = eps;
    return cuda_status(launch_bwd_simt(p, st));
}
}  // namespace

extern "C" {

diffattn_status diffattn_bwd(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                             diffattn_tensor v, const void* dy, const float* norm_weight, int B, int H, int N, int d,
                             int Dv, int causal, float lambda, float lambda_init, float eps, int in_dtype, float* dq1,
                             float* dq2, float* dk1, float* dk2, float* dv, float* dlambda, float* dnorm_weight,
                             void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(q1, q2, k1, k2, v, dy, norm_weight, B, H, N, d, Dv, causal, lambda, lambda_init, eps, in_dtype,
                    dq1, dq2, dk1, dk2, dv, dlambda, dnorm_weight, workspace, workspace_bytes, stream, nullptr);
}

diffattn_status diffattn_bwd_saved(diffattn_tensor q1, diffattn_tensor q2, diffattn_tensor k1, diffattn_tensor k2,
                                   diffattn_tensor v, const void* dy, const float* norm_weight, int B, int H, int N,
                                   int d, int Dv, int causal, float lambda, float lambda_init, float eps, int in_dtype,
                                   const void* saved, size_t saved_bytes, float* dq1, float* dq2, float* dk1,
                                   float* dk2, float* dv, float* dlambda, float* dnorm_weight, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    if (in_dtype == DIFFATTN_F32) return DIFFATTN_ERR_UNSUPPORTED;
    if (B > 0 && H > 0 && N > 0) {
        if (!(d == 64 && Dv == 128)) return DIFFATTN_ERR_UNSUPPORTED;
        if (!saved_ok(saved, saved_bytes, B, H, N, Dv)) return DIFFATTN_ERR_INVALID_ARG;
    }
    return bwd_impl(q1, q2, k1, k2, v, dy, norm_weight, B, H, N, d, Dv, causal, lambda, lambda_init, eps, in_dtype,
                    dq1, dq2, dk1, dk2, dv, dlambda, dnorm_weight, workspace, workspace_bytes, stream,
                    saved);
}

diffattn_status diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2, const float* lk2, int d,
                                    float dlambda, float* dlq1, float* dlk1, float* dlq2, float* dlk2) {
    if (!lq1 || !lk1 || !lq2 || !lk2 || !dlq1 || !dlk1 || !dlq2 || !dlk2 || d < 1 || !isfinite(dlambda))
        return DIFFATTN_ERR_INVALID_ARG;
    double d1 = 0.0, d2 = 0.0;
    for (int i = 0; i < d; ++i) {
        d1 += (double)lq1[i] * (double)lk1[i];
        d2 += (double)lq2[i] * (double)lk2[i];
    }
    const double e1 = exp(d1), e2 = exp(d2);
    if (!isfinite(e1) || !isfinite(e2)) return DIFFATTN_ERR_INVALID_ARG;
    for (int i = 0; i < d; ++i) {
        const double a = lq1[i], b = lk1[i], c = lq2[i], e = lk2[i];
        dlq1[i] = (float)(dlambda * e1 * b);
        dlk1[i] = (float)(dlambda * e1 * a);
        dlq2[i] = (float)(-dlambda * e2 * e);
        dlk2[i] = (float)(-dlambda * e2 * c);
    }
    return DIFFATTN_OK;
}

diffattn_status diffattn_add_rmsnorm(const void* x, int x_dtype, const float* z, float* y_out, void* n_out,
                                     int n_dtype, const float* weight, int M, int N, float eps, void* stream) {
    if (M < 0 || N < 8 || N % 8 || (x_dtype != DIFFATTN_F32 && x_dtype != DIFFATTN_BF16)) return DIFFATTN_ERR_INVALID_ARG;
    if (n_dtype != DIFFATTN_BF16 && n_dtype != DIFFATTN_F16) return DIFFATTN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return DIFFATTN_ERR_INVALID_ARG;
    if (M == 0) return DIFFATTN_OK;
    if (!x || !aligned16(x) || (z && !aligned16(z)) || (y_out && !aligned16(y_out)) || (n_out && !aligned16(n_out)) ||
        (weight && !aligned16(weight)))
        return DIFFATTN_ERR_INVALID_ARG;
    AddNormParams p{};
    p.x = x;
    p.x_f32 = x_dtype == DIFFATTN_F32;
    p.z = z;
    p.y_out = y_out;
    p.n_out = n_out;
    p.n_f16 = n_dtype == DIFFATTN_F16;
    p.weight = weight;
    p.M = M; p.N = N; p.eps = eps;
    return cuda_status(launch_add_rmsnorm(p, static_cast<cudaStream_t>(stream)));
}

diffattn_status diffattn_swiglu(const void* gate_up, void* h_out, int h_dtype, int M, int H, void* stream) {
    if (M < 0 || H < 8 || H % 8 || (h_dtype != DIFFATTN_BF16 && h_dtype != DIFFATTN_F16)) return DIFFATTN_ERR_INVALID_ARG;
    if (M == 0) return DIFFATTN_OK;
    if (!gate_up || !h_out || !aligned16(gate_up) || !aligned16(h_out)) return DIFFATTN_ERR_INVALID_ARG;
    return cuda_status(
        launch_swiglu(gate_up, h_out, h_dtype == DIFFATTN_F16, M, H, static_cast<cudaStream_t>(stream)));
}

namespace {
bool valid_scale(float s) { return isfinite(s) && s > 0.f; }

diffattn_status kv_append(bool fp8, const float* scales, const void* k1_new, const void* k2_new, const void* v_new,
                          diffattn_tensor k1_pages, diffattn_tensor k2_pages, diffattn_tensor v_pages,
                          const int32_t* block_table, int max_pages, int num_pages, const int32_t* seq_lens, int B,
                          int H_kv, int d, int Dv, void* stream) {
    if (B < 0 || H_kv < 0 || d < 8 || Dv < 8 || (d % 8) || (Dv % 8) || max_pages < 1 || num_pages < 1)
        return DIFFATTN_ERR_INVALID_ARG;
    if (fp8 && !(valid_scale(scales[0]) && valid_scale(scales[1]) && valid_scale(scales[2])))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B == 0 || H_kv == 0) return DIFFATTN_OK;
    if (!k1_new || !k2_new || !v_new || !aligned16(k1_new) || !aligned16(k2_new) || !aligned16(v_new) ||
        !block_table || !seq_lens)
        return DIFFATTN_ERR_INVALID_ARG;
    const int eb = fp8 ? 1 : 2;
    if (!check_operand(k1_pages, d, eb) || !check_operand(k2_pages, d, eb) || !check_operand(v_pages, Dv, eb))
        return DIFFATTN_ERR_INVALID_ARG;
    if (k1_pages.stride_b != k2_pages.stride_b || k1_pages.stride_h != k2_pages.stride_h ||
        k1_pages.stride_n != k2_pages.stride_n)
        return DIFFATTN_ERR_INVALID_ARG;
    KvAppendParams p{};
    p.k1_new = k1_new; p.k2_new = k2_new; p.v_new = v_new;
    p.k1_pages = const_cast<void*>(k1_pages.ptr);
    p.k2_pages = const_cast<void*>(k2_pages.ptr);
    p.v_pages = const_cast<void*>(v_pages.ptr);
    p.k_stride_page = k1_pages.stride_b; p.k_stride_h = k1_pages.stride_h; p.k_stride_row = k1_pages.stride_n;
    p.v_stride_page = v_pages.stride_b; p.v_stride_h = v_pages.stride_h; p.v_stride_row = v_pages.stride_n;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.max_pages = max_pages; p.num_pages = num_pages;
    p.B = B; p.H_kv = H_kv; p.d = d; p.Dv = Dv;
    p.fp8 = fp8;
    if (fp8) {
        p.k1_scale = scales[0]; p.k2_scale = scales[1]; p.v_scale = scales[2];
    }
    return cuda_status(launch_kv_append_paged(p, static_cast<cudaStream_t>(stream)));
}
}  // namespace

diffattn_status diffattn_kv_append_paged(const void* k1_new, const void* k2_new, const void* v_new,
                                         diffattn_tensor k1_pages, diffattn_tensor k2_pages, diffattn_tensor v_pages,
                                         const int32_t* block_table, int max_pages, int num_pages,
                                         const int32_t* seq_lens, int B, int H_kv, int d, int Dv, void* stream) {
    return kv_append(false, nullptr, k1_new, k2_new, v_new, k1_pages, k2_pages, v_pages, block_table, max_pages,
                     num_pages, seq_lens, B, H_kv, d, Dv, stream);
}

diffattn_status diffattn_kv_append_paged_fp8(const void* k1_new, const void* k2_new, const void* v_new,
                                             diffattn_tensor k1_pages, diffattn_tensor k2_pages,
                                             diffattn_tensor v_pages, const int32_t* block_table, int max_pages,
                                             int num_pages, const int32_t* seq_lens, int B, int H_kv, int d, int Dv,
                                             float k1_scale, float k2_scale, float v_scale, void* stream) {
    const float scales[3] = {k1_scale, k2_scale, v_scale};
    return kv_append(true, scales, k1_new, k2_new, v_new, k1_pages, k2_pages, v_pages, block_table, max_pages,
                     num_pages, seq_lens, B, H_kv, d, Dv, stream);
}

namespace {
diffattn_status decode_paged(bool fp8, const float* scales, const void* q1, const void* q2, diffattn_tensor k1_pages,
                             diffattn_tensor k2_pages, diffattn_tensor v_pages, const int32_t* block_table,
                             int max_pages, int num_pages, const int32_t* seq_lens, int L, void* out,
                             const float* norm_weight, int B, int H, int kv_group, int d, int Dv, float lambda,
                             float lambda_init, float eps, int num_splits, int out_dtype, void* workspace,
                             size_t workspace_bytes, void* stream) {
    if (B < 0 || H < 0 || L < 1 || d < 1 || Dv < 1 || num_splits < 0 || num_splits > 256 || kv_group < 1 ||
        max_pages < 1 || num_pages < 1)
        return DIFFATTN_ERR_INVALID_ARG;
    if (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16) return DIFFATTN_ERR_INVALID_ARG;
    if (!isfinite(lambda) || !isfinite(lambda_init) || !(eps >= 0.f) || !isfinite(eps))
        return DIFFATTN_ERR_INVALID_ARG;
    if (fp8 && !(valid_scale(scales[0]) && valid_scale(scales[1]) && valid_scale(scales[2])))
        return DIFFATTN_ERR_INVALID_ARG;
    if (B == 0 || H == 0) return DIFFATTN_OK;
    const int stage = decode_keys_per_stage(d);  // one page = one stage of keys
    if (H % kv_group != 0 || L > (int64_t)stage * max_pages) return DIFFATTN_ERR_INVALID_ARG;
    if (!q1 || !q2 || !aligned16(q1) || !aligned16(q2) || !out || !aligned16(out) || !block_table || !seq_lens)
        return DIFFATTN_ERR_INVALID_ARG;
    const int eb = fp8 ? 1 : 2;
    if (!check_operand(k1_pages, d, eb) || !check_operand(k2_pages, d, eb) || !check_operand(v_pages, Dv, eb))
        return DIFFATTN_ERR_INVALID_ARG;
    if (norm_weight != nullptr && !aligned16(norm_weight)) return DIFFATTN_ERR_INVALID_ARG;
    if (!((d == 64 && Dv == 128) || (d == 128 && Dv == 256))) return DIFFATTN_ERR_UNSUPPORTED;
    DecodeParams p{};
    decode_geometry(B, H, L, d, num_splits, &p.num_splits, &p.keys_per_split, fp8);
    const size_t need = decode_ws_bytes(B, H, p.num_splits, Dv);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    const int H_kv = H / kv_group;
    bool ok;
    if (fp8) {
        // Whole key rows in one box: 64 bytes unswizzled (d = 64) or 128 bytes swizzled (d = 128).
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        const CUtensorMapSwizzle ksw = d == 64 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
        ok = encode_4d(&p.tm_k1, k1_pages, d, stage, H_kv, num_pages, d, stage, ksw, u8) &&
             encode_4d(&p.tm_k2, k2_pages, d, stage, H_kv, num_pages, d, stage, ksw, u8) &&
             encode_4d(&p.tm_v, v_pages, Dv, stage, H_kv, num_pages, Dv, stage, CU_TENSOR_MAP_SWIZZLE_NONE, u8);
        p.kv_fp8 = 1;
        p.k1_scale = scales[0]; p.k2_scale = scales[1]; p.v_scale = scales[2];
    } else {
        ok = encode_4d(&p.tm_k1, k1_pages, d, stage, H_kv, num_pages, 64, stage, CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_4d(&p.tm_k2, k2_pages, d, stage, H_kv, num_pages, 64, stage, CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_4d(&p.tm_v, v_pages, Dv, stage, H_kv, num_pages, Dv, stage, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return DIFFATTN_ERR_INVALID_ARG;
    p.q1 = q1;
    p.q2 = q2;
    p.seq_lens = seq_lens;
    p.L = L;
    p.out = out;
    p.out_bf16 = out_dtype == DIFFATTN_BF16;
    p.norm_w = norm_weight;
    p.B = B; p.H = H; p.d = d; p.Dv = Dv;
    p.lambda = lambda; p.lambda_init = lambda_init; p.eps = eps;
    p.block_table = block_table;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.kv_group = kv_group;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.err = err_word(workspace);
    p.part_stats = reinterpret_cast<float*>(ws + kControlBytes);
    p.part_o = p.part_stats + (size_t)B * H * p.num_splits * 4;
    return cuda_status(launch_decode_bf16(p, static_cast<cudaStream_t>(stream)));
}
}  // namespace

diffattn_status diffattn_decode_paged(const void* q1, const void* q2, diffattn_tensor k1_pages,
                                      diffattn_tensor k2_pages, diffattn_tensor v_pages, const int32_t* block_table,
                                      int max_pages, int num_pages, const int32_t* seq_lens, int L, void* out,
                                      const float* norm_weight, int B, int H, int kv_group, int d, int Dv,
                                      float lambda, float lambda_init, float eps, int num_splits, int out_dtype,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    return decode_paged(false, nullptr, q1, q2, k1_pages, k2_pages, v_pages, block_table, max_pages, num_pages,
                        seq_lens, L, out, norm_weight, B, H, kv_group, d, Dv, lambda, lambda_init, eps, num_splits,
                        out_dtype, workspace, workspace_bytes, stream);
}

diffattn_status diffattn_decode_paged_fp8(const void* q1, const void* q2, diffattn_tensor k1_pages,
                                          diffattn_tensor k2_pages, diffattn_tensor v_pages,
                                          const int32_t* block_table, int max_pages, int num_pages,
                                          const int32_t* seq_lens, int L, void* out, const float* norm_weight, int B,
                                          int H, int kv_group, int d, int Dv, float lambda, float lambda_init,
                                          float eps, float k1_scale, float k2_scale, float v_scale, int num_splits,
                                          int out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    const float scales[3] = {k1_scale, k2_scale, v_scale};
    return decode_paged(true, scales, q1, q2, k1_pages, k2_pages, v_pages, block_table, max_pages, num_pages,
                        seq_lens, L, out, norm_weight, B, H, kv_group, d, Dv, lambda, lambda_init, eps, num_splits,
                        out_dtype, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- decode without caller workspace
// Scratch for diffattn_decode_noalloc: error word, then the split partial
// states, exactly as in a diffattn_decode workspace. Host code must not use the
// symbol as an address; it looks the device address up per device.
static __device__ __align__(256) uint8_t g_decode_scratch[DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES];

}  // extern "C"

namespace {
// Device address of g_decode_scratch in the current device's context. It is
// looked up on every call rather than cached: a device reset reloads the
// module, and the array may then sit at another address. Once the module is
// loaded on a device the lookup costs little; the first lookup on a device
// loads it, which is why the first call must precede any stream capture.
void* decode_scratch_address() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
    return ptr;
}
}  // namespace

extern "C" {

diffattn_status diffattn_decode_noalloc(const void* q1, const void* q2, diffattn_tensor k1_cache,
                                        diffattn_tensor k2_cache, diffattn_tensor v_cache, const int32_t* seq_lens,
                                        int L, void* out, const float* norm_weight, int B, int H, int d, int Dv,
                                        float lambda, float lambda_init, float eps, int num_splits, int out_dtype,
                                        void* stream) {
    // The argument checks come first, so a bad call writes nothing to the shared
    // scratch (whose error word a call in flight on another stream may own).
    const diffattn_status chk = decode_check_args(q1, q2, k1_cache, k2_cache, v_cache, L, out, norm_weight, B, H, d,
                                                  Dv, lambda, lambda_init, eps, num_splits, out_dtype);
    if (chk != DIFFATTN_OK || B == 0 || H == 0) return chk;
    int S, kps;  // the bf16-cache geometry diffattn_decode will use
    decode_geometry(B, H, L, d, num_splits, &S, &kps, false);
    if (decode_ws_bytes(B, H, S, Dv) > sizeof(g_decode_scratch)) return DIFFATTN_ERR_WORKSPACE;
    void* scratch = decode_scratch_address();
    if (scratch == nullptr) return DIFFATTN_ERR_CUDA;
    // The error word must start at zero; the partial states are fully rewritten by the split kernel.
    if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    return diffattn_decode(q1, q2, k1_cache, k2_cache, v_cache, seq_lens, L, out, norm_weight, B, H, d, Dv, lambda,
                           lambda_init, eps, num_splits, out_dtype, scratch, sizeof(g_decode_scratch), stream);
}

diffattn_status diffattn_decode_noalloc_read_error(void* stream, int32_t* device_code) {
    if (!device_code) return DIFFATTN_ERR_INVALID_ARG;
    void* scratch = decode_scratch_address();
    if (scratch == nullptr) return DIFFATTN_ERR_CUDA;
    return diffattn_read_error(scratch, stream, device_code);
}

diffattn_status diffattn_gemm_workspace_size(int M, int N, int K, size_t* bytes) {
    if (!bytes || M < 0 || N < 0 || K < 0) return DIFFATTN_ERR_INVALID_ARG;
    *bytes = kControlBytes;
    return DIFFATTN_OK;
}

namespace {
// Checks shared by the GEMM entry points; fills the operand maps and the map of the
// output C, which has out_cols columns (N, or N / 2 for the SwiGLU epilogue).
diffattn_status gemm_setup(GemmParams& p, bool ab_f16, const void* A, const void* W, void* C, int M, int N, int K,
                           int out_cols, int64_t lda, int64_t ldw, int64_t ldc, int out_dtype, void* workspace,
                           size_t workspace_bytes) {
    if (M < 1 || N < 1 || K < 1) return DIFFATTN_ERR_INVALID_ARG;
    if (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16 && out_dtype != DIFFATTN_F16)
        return DIFFATTN_ERR_INVALID_ARG;
    if (!A || !W || !C || !aligned16(A) || !aligned16(W) || !aligned16(C)) return DIFFATTN_ERR_INVALID_ARG;
    const int cq = out_dtype == DIFFATTN_F32 ? 4 : 8;
    if (lda < K || lda % 8 || ldw < N || ldw % 8 || ldc < out_cols || ldc % cq || N % 8 || out_cols % 8)
        return DIFFATTN_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < kControlBytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    if (!encode_2d(&p.tm_a, A, K, M, lda, kGemmBK, kGemmBM, ab_f16) ||
        !encode_2d(&p.tm_w, W, N, K, ldw, 64, kGemmBK, ab_f16))
        return DIFFATTN_ERR_INVALID_ARG;
    {
        // Output map for the epilogue's TMA stores: 128-byte x 32-row boxes.
        auto enc = tensor_map_encoder();
        const int eb = out_dtype == DIFFATTN_F32 ? 4 : 2;
        const CUtensorMapDataType dt = out_dtype == DIFFATTN_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : out_dtype == DIFFATTN_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        cuuint64_t dims[2] = {(cuuint64_t)out_cols, (cuuint64_t)M};
        cuuint64_t strides[1] = {(cuuint64_t)(ldc * eb)};
        cuuint32_t box[2] = {(cuuint32_t)(128 / eb), 32};
        cuuint32_t es[2] = {1, 1};
        if (!enc || enc(&p.tm_c, dt, 2, C, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DIFFATTN_ERR_INVALID_ARG;
    }
    p.C = C;
    p.ldc = ldc;
    p.M = M; p.N = N; p.K = K;
    p.out_bf16 = out_dtype == DIFFATTN_BF16;
    p.out_f16 = out_dtype == DIFFATTN_F16;
    p.ab_f16 = ab_f16;
    p.err = err_word(workspace);
    return DIFFATTN_OK;
}

diffattn_status gemm_16bit(bool ab_f16, const void* A, const void* W, void* C, int M, int N, int K, int64_t lda,
                           int64_t ldw, int64_t ldc, int out_dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
    GemmParams p{};
    const diffattn_status st =
        gemm_setup(p, ab_f16, A, W, C, M, N, K, N, lda, ldw, ldc, out_dtype, workspace, workspace_bytes);
    if (st != DIFFATTN_OK) return st;
    return cuda_status(launch_gemm_bf16(p, static_cast<cudaStream_t>(stream)));
}

bool is16(int dtype) { return dtype == DIFFATTN_BF16 || dtype == DIFFATTN_F16; }
}  // namespace

diffattn_status diffattn_gemm_residual(const void* A, const void* W, const void* R, float* C, void* C16,
                                       const float* c16_gain, float* row_sq, int M, int N, int K, int64_t lda,
                                       int64_t ldw, int64_t ldr, int64_t ldc, int64_t ldc16, int ab_dtype,
                                       int r_dtype, int c16_dtype, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (!is16(ab_dtype) || !(r_dtype == DIFFATTN_F32 || is16(r_dtype))) return DIFFATTN_ERR_INVALID_ARG;
    if (N % kGemmBN) return DIFFATTN_ERR_INVALID_ARG;
    const int rq = r_dtype == DIFFATTN_F32 ? 4 : 8;
    if (!R || !aligned16(R) || ldr < N || ldr % rq) return DIFFATTN_ERR_INVALID_ARG;
    if (C16 && (!is16(c16_dtype) || !aligned16(C16) || ldc16 < N || ldc16 % 8)) return DIFFATTN_ERR_INVALID_ARG;
    if (c16_gain && !C16) return DIFFATTN_ERR_INVALID_ARG;
    GemmParams p{};
    const diffattn_status st = gemm_setup(p, ab_dtype == DIFFATTN_F16, A, W, C, M, N, K, N, lda, ldw, ldc,
                                          DIFFATTN_F32, workspace, workspace_bytes);
    if (st != DIFFATTN_OK) return st;
    p.mode = 1;
    p.resid = R;
    p.ld_r = ldr;
    p.r_dtype = r_dtype == DIFFATTN_F32 ? 0 : (r_dtype == DIFFATTN_BF16 ? 1 : 2);
    p.c16 = C16;
    p.ld_c16 = ldc16;
    p.c16_f16 = c16_dtype == DIFFATTN_F16;
    p.c16_gain = c16_gain;
    p.row_sq = row_sq;
    return cuda_status(launch_gemm_bf16(p, static_cast<cudaStream_t>(stream)));
}

diffattn_status diffattn_gemm_swiglu(const void* A, const void* W_gu, void* H, const float* row_sq, int n_sq,
                                     float sq_count, float eps, int M, int F, int K, int64_t lda, int64_t ldw,
                                     int64_t ldh, int ab_dtype, int h_dtype, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    if (!is16(ab_dtype) || !is16(h_dtype)) return DIFFATTN_ERR_INVALID_ARG;
    if (F < 1 || F % (kGemmBN / 2)) return DIFFATTN_ERR_INVALID_ARG;
    if (row_sq && (n_sq < 1 || !(sq_count > 0.f) || !(eps >= 0.f) || !std::isfinite(sq_count) || !std::isfinite(eps)))
        return DIFFATTN_ERR_INVALID_ARG;
    GemmParams p{};
    const diffattn_status st = gemm_setup(p, ab_dtype == DIFFATTN_F16, A, W_gu, H, M, 2 * F, K, F, lda, ldw, ldh,
                                          h_dtype, workspace, workspace_bytes);
    if (st != DIFFATTN_OK) return st;
    p.mode = 2;
    p.row_sq_in = row_sq;
    p.n_sq = row_sq ? n_sq : 0;
    p.sq_count = sq_count;
    p.eps = eps;
    return cuda_status(launch_gemm_bf16(p, static_cast<cudaStream_t>(stream)));
}

diffattn_status diffattn_gemm_bf16(const void* A, const void* W, void* C, int M, int N, int K, int64_t lda,
                                   int64_t ldw, int64_t ldc, int out_dtype, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    return gemm_16bit(false, A, W, C, M, N, K, lda, ldw, ldc, out_dtype, workspace, workspace_bytes, stream);
}

diffattn_status diffattn_gemm_f16(const void* A, const void* W, void* C, int M, int N, int K, int64_t lda,
                                  int64_t ldw, int64_t ldc, int out_dtype, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    return gemm_16bit(true, A, W, C, M, N, K, lda, ldw, ldc, out_dtype, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// End-to-end prefill from host buffers: the batch in pieces, each piece's copies
// in, prefill and copy back on three library streams so that they overlap.
// ---------------------------------------------------------------------------
}  // extern "C"
namespace {
constexpr int kMaxHostChunks = 16;
struct HostPipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in_done[kMaxHostChunks], run_done[kMaxHostChunks];
};
std::mutex g_pipe_mu;  // one pipelined call at a time (the streams and events are shared)
HostPipe g_pipe[64];

// The streams and events of the current device, created on first use.
HostPipe* host_pipe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    HostPipe& hp = g_pipe[dev];
    if (!hp.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.s_run, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, ef) != cudaSuccess || cudaEventCreateWithFlags(&hp.done, ef) != cudaSuccess)
            return nullptr;
        for (int i = 0; i < kMaxHostChunks; ++i)
            if (cudaEventCreateWithFlags(&hp.in_done[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.run_done[i], ef) != cudaSuccess)
                return nullptr;
        hp.ready = true;
    }
    return &hp;
}

// Byte offsets of the pieces of the device buffer: the workspace (error word) first,
// then Q1, Q2, K1, K2, V ([B, H, N, width] contiguous) and the output [B, N, H, Dv].
struct HostLayout {
    size_t in[5], out, total;
};
HostLayout host_layout(int B, int H, int N, int d, int Dv, int in_eb, int out_eb) {
    HostLayout L{};
    size_t off = round256(kControlBytes);
    for (int i = 0; i < 5; ++i) {
        L.in[i] = off;
        off += round256((size_t)B * H * N * (i == 4 ? Dv : d) * in_eb);
    }
    L.out = off;
    off += round256((size_t)B * N * H * Dv * out_eb);
    L.total = off;
    return L;
}
int dtype_bytes(int dt) { return dt == DIFFATTN_F32 ? 4 : 2; }
}  // namespace
extern "C" {

diffattn_status diffattn_fwd_host_buffer_size(int B, int H, int N, int d, int Dv, int in_dtype, int out_dtype,
                                              size_t* bytes) {
    if (!bytes || B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1) return DIFFATTN_ERR_INVALID_ARG;
    if ((in_dtype != DIFFATTN_F32 && in_dtype != DIFFATTN_BF16 && in_dtype != DIFFATTN_F16) ||
        (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16 && out_dtype != DIFFATTN_F16))
        return DIFFATTN_ERR_INVALID_ARG;
    *bytes = host_layout(B, H, N, d, Dv, dtype_bytes(in_dtype), dtype_bytes(out_dtype)).total;
    return DIFFATTN_OK;
}

diffattn_status diffattn_fwd_host(const void* q1, const void* q2, const void* k1, const void* k2, const void* v,
                                  void* out, const float* norm_weight, int B, int H, int N, int d, int Dv, int causal,
                                  float lambda, float lambda_init, float eps, int in_dtype, int out_dtype, int chunks,
                                  void* device_buffer, size_t device_buffer_bytes, void* stream) {
    if (!q1 || !q2 || !k1 || !k2 || !v || !out || B < 0 || H < 0 || N < 0 || d < 1 || Dv < 1 || chunks < 0 ||
        chunks > kMaxHostChunks)
        return DIFFATTN_ERR_INVALID_ARG;
    if ((in_dtype != DIFFATTN_F32 && in_dtype != DIFFATTN_BF16 && in_dtype != DIFFATTN_F16) ||
        (out_dtype != DIFFATTN_F32 && out_dtype != DIFFATTN_BF16 && out_dtype != DIFFATTN_F16))
        return DIFFATTN_ERR_INVALID_ARG;
    const int ieb = dtype_bytes(in_dtype), oeb = dtype_bytes(out_dtype);
    const HostLayout L = host_layout(B, H, N, d, Dv, ieb, oeb);
    if (device_buffer == nullptr || device_buffer_bytes < L.total || (reinterpret_cast<uintptr_t>(device_buffer) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    if (B == 0 || H == 0 || N == 0) return DIFFATTN_OK;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe* hp = host_pipe();
    if (!hp) return DIFFATTN_ERR_CUDA;
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    uint8_t* dev = static_cast<uint8_t*>(device_buffer);
    const void* host_in[5] = {q1, q2, k1, k2, v};
    // Pieces are head ranges within one batch entry: (b, h0 .. h1). Their inputs are contiguous
    // in the [B, H, N, *] buffers; each piece's output goes to its own contiguous [N, h1-h0, Dv]
    // slice of the device output region and back with one pitched copy into [B, N, H, Dv].
    // Default 4 pieces: smaller ones were measured slower (each pays its tensor-map encodes and
    // launch, and pitched copies of short rows), so head ranges only split small batches.
    const int want = chunks > 0 ? chunks : 4;
    const int per_b = std::max(1, std::min(H, (want + B - 1) / B));  // pieces per batch entry
    const int hg = (H + per_b - 1) / per_b;                           // heads per piece
    // Everything is ordered after the caller's earlier work, and the caller's later work after it.
    if (cudaEventRecord(hp->start, caller) != cudaSuccess || cudaStreamWaitEvent(hp->s_in, hp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->s_run, hp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->s_out, hp->start, 0) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    int i = 0;
    for (int b = 0; b < B; ++b) {
        for (int h0 = 0; h0 < H; h0 += hg, ++i) {
            const int h1 = std::min(H, h0 + hg), nh = h1 - h0;
            // Events are reused after 16 pieces: a stream wait binds to the record current when the
            // wait is enqueued, so recording the event again later does not affect it.
            const int ev = i % kMaxHostChunks;
            const int64_t unit0 = (int64_t)b * H + h0;  // first (b, h) of the piece
            diffattn_tensor ts[5];
            for (int t = 0; t < 5; ++t) {
                const int w = t == 4 ? Dv : d;
                const size_t per_h = (size_t)N * w * ieb;
                if (cudaMemcpyAsync(dev + L.in[t] + unit0 * per_h, static_cast<const uint8_t*>(host_in[t]) + unit0 * per_h,
                                    nh * per_h, cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess)
                    return DIFFATTN_ERR_CUDA;
                ts[t] = diffattn_tensor{dev + L.in[t] + unit0 * per_h, (int64_t)H * N * w, (int64_t)N * w, w};
            }
            if (cudaEventRecord(hp->in_done[ev], hp->s_in) != cudaSuccess ||
                cudaStreamWaitEvent(hp->s_run, hp->in_done[ev], 0) != cudaSuccess)
                return DIFFATTN_ERR_CUDA;
            uint8_t* dout = dev + L.out + (size_t)unit0 * N * Dv * oeb;  // [N, nh, Dv]
            const diffattn_status st = diffattn_fwd(ts[0], ts[1], ts[2], ts[3], ts[4], dout, norm_weight, 1, nh, N, d,
                                                    Dv, causal, lambda, lambda_init, eps, in_dtype, out_dtype, dev,
                                                    kControlBytes, hp->s_run);
            if (st != DIFFATTN_OK) return st;
            const size_t row = (size_t)nh * Dv * oeb;
            if (cudaEventRecord(hp->run_done[ev], hp->s_run) != cudaSuccess ||
                cudaStreamWaitEvent(hp->s_out, hp->run_done[ev], 0) != cudaSuccess ||
                cudaMemcpy2DAsync(static_cast<uint8_t*>(out) + ((size_t)b * N * H + h0) * Dv * oeb,
                                  (size_t)H * Dv * oeb, dout, row, row, N, cudaMemcpyDeviceToHost,
                                  hp->s_out) != cudaSuccess)
                return DIFFATTN_ERR_CUDA;
        }
    }
    // The last copy back follows every prefill, which follows every copy in.
    if (cudaEventRecord(hp->done, hp->s_out) != cudaSuccess || cudaStreamWaitEvent(caller, hp->done, 0) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    return DIFFATTN_OK;
}

diffattn_status diffattn_selftest_timeout(void* workspace, size_t workspace_bytes, void* stream) {
    if (workspace == nullptr || workspace_bytes < kControlBytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DIFFATTN_ERR_WORKSPACE;
    return cuda_status(launch_selftest_timeout(err_word(workspace), static_cast<cudaStream_t>(stream)));
}

diffattn_status diffattn_read_error(void* workspace, void* stream, int32_t* device_code) {
    if (!workspace || !device_code) return DIFFATTN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t code = 0;
    if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    *device_code = code;
    if (code == 0) return DIFFATTN_OK;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return DIFFATTN_ERR_CUDA;
    return DIFFATTN_ERR_TIMEOUT;
}

}  // extern "C"
