// gdn_api.cu -- the C ABI declared in include/gdn.h: argument checks and
// dispatch to the kernels. Nothing here allocates or synchronises (except
// gdn_device_error, which is documented to).
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "gdn_common.cuh"

namespace gdn {
void *decode_error_word();
cudaError_t launch_conv_step(const float *, const void *, void *, void *, int, gdn_dtype, cudaStream_t);
cudaError_t launch_decode_step(const gdn_params *, const void *, const void *, const void *, const void *,
                               void *, float *, void *, int, gdn_dtype, gdn_dtype, cudaStream_t);
cudaError_t launch_decode_multi(const gdn_params *, const void *, const void *, const void *, const void *,
                                void *, float *, void *, int, int, gdn_dtype, gdn_dtype, cudaStream_t);
void *multi_error_word();
cudaError_t launch_out_proj(const void *x, const void *w, void *y, int M, gdn_dtype out_dt, cudaStream_t s);
void *gemm_error_word();
cudaError_t launch_gated_out_proj(const float *norm_w, float eps, const void *y, const void *z, const void *w,
                                  void *out, int M, gdn_dtype act, gdn_dtype out_dt, cudaStream_t s);
void *gproj_error_word();
cudaError_t launch_in_proj(const void *h, const void *w_in, void *qkv, void *z, void *alpha, void *beta, int M,
                           gdn_dtype act, cudaStream_t s);
size_t scan_workspace_bytes(int T_total);
cudaError_t launch_prefill_scan(const gdn_params *, const void *, const void *, const void *, const void *,
                                const int32_t *, int, int, const void *, void *, const float *, float *,
                                void *, gdn_dtype, gdn_dtype, void *, cudaStream_t);
size_t chunk_workspace_bytes(int N, int T_total);
size_t chunk_min_workspace_bytes(int N);
cudaError_t launch_prefill_chunked(const gdn_params *, const void *, const void *, const void *, const void *,
                                   const int32_t *, int, int, const void *, void *, const float *, float *, void *,
                                   gdn_dtype, void *, size_t, cudaStream_t, const void *xhat_ext);
void *chunk_error_word();
cudaError_t launch_in_proj_conv(const float *conv_w, float l2_eps, const void *h, const void *w_in,
                                const int32_t *cu, int N, int M, const void *cs_in, void *cs_out, void *xhat,
                                void *z, void *alpha, void *beta, cudaStream_t s);
void *inconv_error_word();
size_t attn_workspace_bytes(int B, int Lmax);
cudaError_t launch_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                               const void *z, void *out, int B, int Lmax, void *ws, gdn_dtype out_dt,
                               cudaStream_t s);
void *attn_error_word();
cudaError_t launch_wait_timeout(cudaStream_t s);
void *selftest_error_word();
}  // namespace gdn

using namespace gdn;

namespace {

thread_local char g_last_error[256] = "";

gdn_status fail(gdn_status s, const char *what)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s", what);
    return s;
}

gdn_status cuda_fail(cudaError_t e, const char *where)
{
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
    return GDN_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
bool ok_opt_ptr(const void *p) { return p == nullptr || aligned16(p); }
bool ok_dtype(gdn_dtype d) { return d == GDN_F32 || d == GDN_BF16; }

gdn_status check_params(const gdn_params *p)
{
    if (p == nullptr) return fail(GDN_ERR_INVALID_ARG, "params is NULL");
    if (!ok_ptr(p->conv_w) || !ok_ptr(p->A_log) || !ok_ptr(p->dt_bias) || !ok_opt_ptr(p->norm_w))
        return fail(GDN_ERR_INVALID_ARG, "a parameter pointer is NULL or not 16-byte aligned");
    if (!(p->norm_eps >= 0.0f) || !(p->l2_eps >= 0.0f))
        return fail(GDN_ERR_INVALID_ARG, "epsilons must be >= 0");
    return GDN_OK;
}

constexpr int MAX_B = 65535;
constexpr int MAX_N = 65535;
constexpr int MAX_T = 1 << 24;
constexpr size_t WS_HEADER = 256;   // keeps the workspace body 256-byte aligned

// chunk_size 0 = library choice: the exact scan for fp32 activations, the
// chunked tensor-core form for bf16 activations.
int resolve_chunk(int chunk_size, gdn_dtype act)
{
    if (chunk_size == 0) return act == GDN_BF16 ? 64 : 1;
    return chunk_size;
}

}  // namespace

namespace gdn {

// Every kernel file keeps its own device error word. gdn_device_error reads and
// clears all of them with one small kernel (an atomic exchange each, so a word
// set while the call runs is either reported now or kept for the next call)
// and one copy of the OR back to the host.
constexpr int N_ERROR_WORDS = 8;
struct ErrorWords {
    unsigned int *p[N_ERROR_WORDS];
};
__device__ unsigned int g_error_any;

__global__ void error_gather_kernel(const ErrorWords w)
{
    if (threadIdx.x != 0) return;
    unsigned int v = 0;
#pragma unroll
    for (int i = 0; i < N_ERROR_WORDS; ++i)
        if (w.p[i]) v |= atomicExch(w.p[i], 0u);
    g_error_any = v;
}

// The words' device addresses, looked up once per device with that device
// current (a host-side symbol is not a device address).
static bool error_words(ErrorWords *out)
{
    constexpr int MAX_DEV = 64;
    static std::mutex mu;
    static ErrorWords cache[MAX_DEV];
    static bool have[MAX_DEV] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        void *(*const fns[N_ERROR_WORDS])() = {decode_error_word, chunk_error_word,    multi_error_word,
                                               gemm_error_word,   attn_error_word,     selftest_error_word,
                                               gproj_error_word,  inconv_error_word};
        for (int i = 0; i < N_ERROR_WORDS; ++i) {
            cache[dev].p[i] = static_cast<unsigned int *>(fns[i]());
            if (cache[dev].p[i] == nullptr) return false;
        }
        have[dev] = true;
    }
    *out = cache[dev];
    return true;
}

// Lets other translation units of the library set the gdn_last_error() text.
void record_error(const char *msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
}  // namespace gdn

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char *gdn_last_error(void) { return g_last_error; }

const char *gdn_status_string(gdn_status s)
{
    switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "GDN_STATUS_UNKNOWN";
}

gdn_status gdn_conv_step(const float *conv_w, const void *qkv_in, void *qkv_out, void *conv_state, int B,
                         gdn_dtype act, void *stream)
{
    if (!ok_dtype(act)) return fail(GDN_ERR_INVALID_ARG, "unknown activation dtype");
    if (B < 0 || B > MAX_B) return fail(GDN_ERR_INVALID_ARG, "B out of range [0, 65535]");
    if (B == 0) return GDN_OK;
    if (!ok_ptr(conv_w) || !ok_ptr(qkv_in) || !ok_ptr(qkv_out) || !ok_ptr(conv_state))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (qkv_in == qkv_out) return fail(GDN_ERR_INVALID_ARG, "qkv_out may not alias qkv_in");
    cudaError_t e = launch_conv_step(conv_w, qkv_in, qkv_out, conv_state, B, act, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_conv_step");
}

gdn_status gdn_decode_step(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                           const void *beta, void *conv_state, float *ssm_state, void *out, int B,
                           gdn_dtype act, gdn_dtype out_dt, void *stream)
{
    if (!ok_dtype(act) || !ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
    if (B < 0 || B > MAX_B) return fail(GDN_ERR_INVALID_ARG, "B out of range [0, 65535]");
    if (B == 0) return GDN_OK;
    gdn_status st = check_params(p);
    if (st != GDN_OK) return st;
    if (!ok_ptr(qkv) || !ok_ptr(z) || !ok_ptr(alpha) || !ok_ptr(beta) || !ok_ptr(conv_state) ||
        !ok_ptr(ssm_state) || !ok_ptr(out))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    cudaError_t e = launch_decode_step(p, qkv, z, alpha, beta, conv_state, ssm_state, out, B, act, out_dt,
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_decode_step");
}

gdn_status gdn_decode_multi(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                            const void *beta, void *conv_state, float *ssm_state, void *out, int B, int T,
                            gdn_dtype act, gdn_dtype out_dt, void *stream)
{
    if (!ok_dtype(act) || !ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
    if (B < 0 || B > MAX_B) return fail(GDN_ERR_INVALID_ARG, "B out of range [0, 65535]");
    if (T < 1 || T > GDN_DECODE_MAX_T) return fail(GDN_ERR_INVALID_ARG, "T out of range [1, GDN_DECODE_MAX_T]");
    if (B == 0) return GDN_OK;
    gdn_status st = check_params(p);
    if (st != GDN_OK) return st;
    if (!ok_ptr(qkv) || !ok_ptr(z) || !ok_ptr(alpha) || !ok_ptr(beta) || !ok_ptr(conv_state) ||
        !ok_ptr(ssm_state) || !ok_ptr(out))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    cudaError_t e = launch_decode_multi(p, qkv, z, alpha, beta, conv_state, ssm_state, out, B, T, act, out_dt,
                                        (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_decode_multi");
}

gdn_status gdn_in_proj(const void *h, const void *w_in, void *qkv, void *z, void *alpha, void *beta, int M,
                       gdn_dtype act, void *stream)
{
    if (!ok_dtype(act)) return fail(GDN_ERR_INVALID_ARG, "unknown activation dtype");
    if (M < 0 || M > (1 << 24)) return fail(GDN_ERR_INVALID_ARG, "M out of range [0, 2^24]");
    if (M == 0) return GDN_OK;
    if (!ok_ptr(h) || !ok_ptr(w_in) || !ok_ptr(qkv) || !ok_ptr(z) || !ok_ptr(alpha) || !ok_ptr(beta))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    cudaError_t e = launch_in_proj(h, w_in, qkv, z, alpha, beta, M, act, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_in_proj");
}

gdn_status gdn_out_proj(const void *x, const void *w, void *y, int M, gdn_dtype out_dt, void *stream)
{
    if (!ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown output dtype");
    if (M < 0 || M > (1 << 24)) return fail(GDN_ERR_INVALID_ARG, "M out of range [0, 2^24]");
    if (M == 0) return GDN_OK;
    if (!ok_ptr(x) || !ok_ptr(w) || !ok_ptr(y))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    cudaError_t e = launch_out_proj(x, w, y, M, out_dt, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_out_proj");
}

gdn_status gdn_gated_out_proj(const float *norm_w, float norm_eps, const void *y, const void *z, const void *w,
                              void *out, int M, gdn_dtype act, gdn_dtype out_dt, void *stream)
{
    if (!ok_dtype(act) || !ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown activation or output dtype");
    if (M < 0 || M > (1 << 24)) return fail(GDN_ERR_INVALID_ARG, "M out of range [0, 2^24]");
    if (M == 0) return GDN_OK;
    if (!ok_ptr(norm_w) || !ok_ptr(y) || !ok_ptr(z) || !ok_ptr(w) || !ok_ptr(out))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (!(norm_eps >= 0.0f)) return fail(GDN_ERR_INVALID_ARG, "norm_eps must be >= 0");
    cudaError_t e = launch_gated_out_proj(norm_w, norm_eps, y, z, w, out, M, act, out_dt, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_gated_out_proj");
}

size_t gdn_attn_decode_workspace_size(int B, int Lmax)
{
    if (B < 1 || B > MAX_B || Lmax < 1 || (long long)B * GDN_ATTN_KV_HEADS * Lmax > (1ll << 30)) return 0;
    return attn_workspace_bytes(B, Lmax);
}

gdn_status gdn_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                           const void *z, void *out, int B, int Lmax, void *workspace, size_t workspace_bytes,
                           gdn_dtype out_dt, void *stream)
{
    if (!ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown output dtype");
    if (B < 0 || B > MAX_B) return fail(GDN_ERR_INVALID_ARG, "B out of range [0, 65535]");
    if (B == 0) return GDN_OK;
    if (Lmax < 1 || (long long)B * GDN_ATTN_KV_HEADS * Lmax > (1ll << 30))
        return fail(GDN_ERR_INVALID_ARG, "Lmax out of range: need 1 <= Lmax and B * 2 * Lmax <= 2^30");
    if (!ok_ptr(q) || !ok_ptr(k_cache) || !ok_ptr(v_cache) || !ok_ptr(z) || !ok_ptr(out))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (ctx_len == nullptr || (reinterpret_cast<uintptr_t>(ctx_len) & 3u) != 0)
        return fail(GDN_ERR_INVALID_ARG, "ctx_len is NULL or not 4-byte aligned");
    if (!ok_ptr(workspace)) return fail(GDN_ERR_WORKSPACE, "workspace is NULL or not 16-byte aligned");
    if (workspace_bytes < attn_workspace_bytes(B, Lmax))
        return fail(GDN_ERR_WORKSPACE, "workspace smaller than gdn_attn_decode_workspace_size(B, Lmax)");
    cudaError_t e = launch_attn_decode(q, k_cache, v_cache, ctx_len, z, out, B, Lmax, workspace, out_dt,
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_attn_decode");
}

size_t gdn_prefill_workspace_size(int N, int T_total, gdn_dtype act, int chunk_size)
{
    if (N < 0 || N > MAX_N || T_total < 0 || T_total > MAX_T || !ok_dtype(act)) return 0;
    const int ch = resolve_chunk(chunk_size, act);
    size_t body = 0;
    if (ch == 1) body = scan_workspace_bytes(T_total);
    else if (ch == 64 && act == GDN_BF16) body = chunk_workspace_bytes(N, T_total);
    else return 0;
    return WS_HEADER + ((body + 255) & ~(size_t)255);
}

gdn_status gdn_prefill(const gdn_params *p, const void *qkv, const void *z, const void *alpha, const void *beta,
                       const int32_t *cu_seqlens, int N, int T_total, const void *conv_state_in,
                       void *conv_state_out, const float *ssm_state_in, float *ssm_state_out, void *out,
                       gdn_dtype act, gdn_dtype out_dt, int chunk_size, void *workspace, size_t ws_bytes,
                       void *stream)
{
    if (!ok_dtype(act) || !ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
    if (N < 0 || N > MAX_N) return fail(GDN_ERR_INVALID_ARG, "N out of range [0, 65535]");
    if (T_total < 0 || T_total > MAX_T) return fail(GDN_ERR_INVALID_ARG, "T_total out of range [0, 2^24]");
    if (N == 0) {
        if (T_total != 0) return fail(GDN_ERR_INVALID_ARG, "T_total > 0 with no sequences");
        return GDN_OK;
    }
    const int ch = resolve_chunk(chunk_size, act);
    if (ch != 1 && ch != 64) return fail(GDN_ERR_UNSUPPORTED, "chunk_size must be 0, 1 or 64");
    if (ch == 64 && act != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "the chunked tensor-core form needs bf16 activations");
    gdn_status st = check_params(p);
    if (st != GDN_OK) return st;
    if (!ok_ptr(cu_seqlens) || (T_total > 0 && (!ok_ptr(qkv) || !ok_ptr(z) || !ok_ptr(alpha) ||
                                                !ok_ptr(beta) || !ok_ptr(out))))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (!ok_opt_ptr(conv_state_in) || !ok_opt_ptr(conv_state_out) || !ok_opt_ptr(ssm_state_in) ||
        !ok_opt_ptr(ssm_state_out))
        return fail(GDN_ERR_INVALID_ARG, "a state pointer is not 16-byte aligned");
    // The exact scan needs its whole workspace. The chunked form runs in windows
    // of the packed tokens sized to the workspace it is given, so any workspace
    // that holds one 64-token window will do.
    const size_t need = ch == 1 ? gdn_prefill_workspace_size(N, T_total, act, ch)
                                : WS_HEADER + ((chunk_min_workspace_bytes(N) + 255) & ~(size_t)255);
    if (workspace == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        snprintf(g_last_error, sizeof(g_last_error),
                 "workspace missing, misaligned (256 B) or too small: %zu bytes given, %zu needed", ws_bytes, need);
        return GDN_ERR_WORKSPACE;
    }
    void *body = static_cast<char *>(workspace) + WS_HEADER;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    if (ch == 1)
        e = launch_prefill_scan(p, qkv, z, alpha, beta, cu_seqlens, N, T_total, conv_state_in, conv_state_out,
                                ssm_state_in, ssm_state_out, out, act, out_dt, body, s);
    else
        e = launch_prefill_chunked(p, qkv, z, alpha, beta, cu_seqlens, N, T_total, conv_state_in, conv_state_out,
                                   ssm_state_in, ssm_state_out, out, out_dt, body, ws_bytes - WS_HEADER, s, nullptr);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_prefill");
}

gdn_status gdn_in_proj_conv(const gdn_params *p, const void *h, const void *w_in, const int32_t *cu_seqlens, int N,
                            int M, const void *conv_state_in, void *conv_state_out, void *xhat, void *z,
                            void *alpha, void *beta, void *stream)
{
    if (N < 0 || N > MAX_N) return fail(GDN_ERR_INVALID_ARG, "N out of range [0, 65535]");
    if (M < 0 || M > MAX_T) return fail(GDN_ERR_INVALID_ARG, "M out of range [0, 2^24]");
    if (N == 0) {
        if (M != 0) return fail(GDN_ERR_INVALID_ARG, "M > 0 with no sequences");
        return GDN_OK;
    }
    if (p == nullptr || !ok_ptr(p->conv_w) || !(p->l2_eps >= 0.0f))
        return fail(GDN_ERR_INVALID_ARG, "params NULL, conv_w NULL or misaligned, or l2_eps < 0");
    if (!ok_ptr(cu_seqlens) || (M > 0 && (!ok_ptr(h) || !ok_ptr(w_in) || !ok_ptr(xhat) || !ok_ptr(z) ||
                                          !ok_ptr(alpha) || !ok_ptr(beta))))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (!ok_opt_ptr(conv_state_in) || !ok_opt_ptr(conv_state_out))
        return fail(GDN_ERR_INVALID_ARG, "a state pointer is not 16-byte aligned");
    const size_t cs_bytes = (size_t)N * (GDN_CONV_K - 1) * GDN_CONV_CHANNELS * 2;
    if (conv_state_in && conv_state_out) {
        const char *i0 = static_cast<const char *>(conv_state_in), *o0 = static_cast<const char *>(conv_state_out);
        if (i0 < o0 + cs_bytes && o0 < i0 + cs_bytes)
            return fail(GDN_ERR_INVALID_ARG, "conv_state_in and conv_state_out overlap");
    }
    cudaError_t e = launch_in_proj_conv(p->conv_w, p->l2_eps, h, w_in, cu_seqlens, N, M, conv_state_in,
                                        conv_state_out, xhat, z, alpha, beta, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_in_proj_conv");
}

gdn_status gdn_prefill_xhat(const gdn_params *p, const void *xhat, const void *z, const void *alpha,
                            const void *beta, const int32_t *cu_seqlens, int N, int T_total,
                            const float *ssm_state_in, float *ssm_state_out, void *out, gdn_dtype out_dt,
                            void *workspace, size_t ws_bytes, void *stream)
{
    if (!ok_dtype(out_dt)) return fail(GDN_ERR_INVALID_ARG, "unknown dtype");
    if (N < 0 || N > MAX_N) return fail(GDN_ERR_INVALID_ARG, "N out of range [0, 65535]");
    if (T_total < 0 || T_total > MAX_T) return fail(GDN_ERR_INVALID_ARG, "T_total out of range [0, 2^24]");
    if (N == 0) {
        if (T_total != 0) return fail(GDN_ERR_INVALID_ARG, "T_total > 0 with no sequences");
        return GDN_OK;
    }
    gdn_status st = check_params(p);
    if (st != GDN_OK) return st;
    if (!ok_ptr(cu_seqlens) || (T_total > 0 && (!ok_ptr(xhat) || !ok_ptr(z) || !ok_ptr(alpha) || !ok_ptr(beta) ||
                                                !ok_ptr(out))))
        return fail(GDN_ERR_INVALID_ARG, "a tensor pointer is NULL or not 16-byte aligned");
    if (!ok_opt_ptr(ssm_state_in) || !ok_opt_ptr(ssm_state_out))
        return fail(GDN_ERR_INVALID_ARG, "a state pointer is not 16-byte aligned");
    const size_t need = WS_HEADER + ((chunk_min_workspace_bytes(N) + 255) & ~(size_t)255);
    if (workspace == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        snprintf(g_last_error, sizeof(g_last_error),
                 "workspace missing, misaligned (256 B) or too small: %zu bytes given, %zu needed", ws_bytes, need);
        return GDN_ERR_WORKSPACE;
    }
    void *body = static_cast<char *>(workspace) + WS_HEADER;
    cudaError_t e = launch_prefill_chunked(p, nullptr, z, alpha, beta, cu_seqlens, N, T_total, nullptr, nullptr,
                                           ssm_state_in, ssm_state_out, out, out_dt, body, ws_bytes - WS_HEADER,
                                           (cudaStream_t)stream, xhat);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_prefill_xhat");
}

gdn_status gdn_device_error(void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    ErrorWords w;
    if (!error_words(&w)) return cuda_fail(cudaGetLastError(), "gdn_device_error: error word lookup");
    unsigned int any = 0;
    error_gather_kernel<<<1, 32, 0, s>>>(w);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&any, g_error_any, sizeof(unsigned int), 0,
                                                        cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "gdn_device_error");
    return any == 0 ? GDN_OK : GDN_ERR_TIMEOUT;
}

gdn_status gdn_get_device_error(void *workspace, void *stream)
{
    (void)workspace;
    return gdn_device_error(stream);
}

gdn_status gdn_selftest_wait_timeout(void *stream)
{
    cudaError_t e = launch_wait_timeout((cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_selftest_wait_timeout");
}

}  // extern "C"
