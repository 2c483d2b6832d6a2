// C ABI of the library (declared in include/csa.h): argument checks,
// workspace planning, TMA descriptor encoding and kernel launches on the
// caller's stream.  No device memory is allocated here.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/csa.h"
#include "common.cuh"
#include "kernels.h"

namespace csa {
__device__ unsigned int g_status = 0;
}

using namespace csa;

namespace {

thread_local char g_msg[512] = "";

csa_status_t fail(csa_status_t st, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

csa_status_t cuda_status(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return CSA_OK;
    return fail(CSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms()
{
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2D row-major [rows, inner] tensor, 128-byte swizzled boxes of
// [box_rows, box_inner] (box_inner * element size = 128 bytes).
csa_status_t make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
                      uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B)
{
    auto enc = tensor_map_encoder();
    if (!enc) return fail(CSA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return CSA_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool tc_indexer_shape(int H_I, int d_I) { return H_I == 64 && d_I == 128; }

csa_status_t check_index_dtypes(csa_dtype_t q_dtype, csa_dtype_t k_dtype, int H_I, int d_I)
{
    const bool f32 = q_dtype == CSA_F32 && k_dtype == CSA_F32;
    const bool bf16 = q_dtype == CSA_BF16 && k_dtype == CSA_BF16;
    const bool fp8 = q_dtype == CSA_E4M3 && (k_dtype == CSA_E4M3 || k_dtype == CSA_E2M1);
    if (!f32 && !bf16 && !fp8)
        return fail(CSA_ERR_UNSUPPORTED, "indexer precision pair (q=%d, k=%d) not supported", q_dtype, k_dtype);
    if (!f32 && !tc_indexer_shape(H_I, d_I))
        return fail(CSA_ERR_UNSUPPORTED, "tensor-core indexer needs H_I=64, d_I=128 (got %d, %d)", H_I, d_I);
    if (f32 && (H_I < 1 || d_I < 1 || (size_t)(H_I * d_I + H_I) * 4 > 200 * 1024))
        return fail(CSA_ERR_UNSUPPORTED, "fp32 indexer shape H_I=%d d_I=%d", H_I, d_I);
    return CSA_OK;
}

// Workspace of the index-scores stage: widened E4M3 keys + row scales for E2M1.
size_t scores_ws_bytes(int B, int N_c, int d_I, csa_dtype_t k_dtype)
{
    if (k_dtype != CSA_E2M1) return 0;
    return align_up((size_t)B * N_c * d_I, 256) + align_up((size_t)B * N_c * 4, 256);
}

// Queries per chunk of csa_index_topk: bounded score buffer (multiple of 4).
int index_chunk_rows(int B, int n_q, int N_c, size_t score_bytes = 4)
{
    const size_t budget = 256ull << 20;
    size_t per_row = (size_t)B * (size_t)(N_c > 0 ? N_c : 1) * score_bytes;
    long long rows = (long long)(budget / per_row);
    if (rows < 4) rows = 4;
    rows &= ~3ll;
    if (rows >= n_q) rows = n_q;
    return (int)(rows > 0 ? rows : 1);
}

// Split-KV plan of the attention kernels.  Decode-shaped calls (few queries
// per sequence) split each query's key set into slices of at least 256 keys
// (a multiple of the tensor-core kernel's 128-key tile) so that one step fills
// the GPU.  The plan depends only on the per-sequence shape, never on the
// batch size, so a sequence's result is bitwise the same at any batch
// position.
struct SplitPlan { int n; int len; };
SplitPlan attn_split_plan(int n_q, long long set_len)
{
    if (n_q > 16 || set_len <= 256) return {1, 1 << 30};
    long long len = 256;
    while ((set_len + len - 1) / len > 64) len += 128;
    return {(int)((set_len + len - 1) / len), (int)len};
}

// wmax non-null: the tensor-core decode kernel also writes each row's warp
// maxima there (the top-k's collection threshold).
csa_status_t run_scores(int B, int n_q, int i_start, int n_q_rows, QPos q_pos0, int m, int N_c, int H_I,
                        int d_I, const void* q_idx, csa_dtype_t q_dtype, const float* q_scale, const void* k_idx,
                        csa_dtype_t k_dtype, const void* k_scale, const float* head_w, bool relu, void* scores,
                        bool sbf16, void* ws, cudaStream_t s, uint32_t* wmax = nullptr, int wmax_ld = 0,
                        uint32_t* zero_words = nullptr, int n_zero = 0)
{
    if (q_dtype == CSA_F32) {
        return cuda_status(launch_indexer_f32(reinterpret_cast<const float*>(q_idx), q_scale, head_w, relu,
                                              reinterpret_cast<const float*>(k_idx),
                                              reinterpret_cast<const float*>(k_scale), scores, sbf16, B, n_q, i_start,
                                              n_q_rows, q_pos0, m, N_c, H_I, d_I, s),
                           "indexer_f32 launch");
    }
    const bool fp8 = q_dtype == CSA_E4M3;
    const void* keys = k_idx;
    const float* ksc = reinterpret_cast<const float*>(k_scale);
    const int T = indexer_group_tokens(n_q_rows);
    // decode groups widen FP4 keys inside the indexer; prefill groups, which
    // read every key tile many times, widen once into the workspace
    const bool kfp4 = k_dtype == CSA_E2M1 && T == 1;
    if (k_dtype == CSA_E2M1 && !kfp4) {
        uint8_t* x8 = reinterpret_cast<uint8_t*>(ws);
        float* S = reinterpret_cast<float*>(x8 + align_up((size_t)B * N_c * d_I, 256));
        csa_status_t st = cuda_status(
            launch_fp4_to_e4m3(reinterpret_cast<const uint8_t*>(k_idx), reinterpret_cast<const uint8_t*>(k_scale),
                               x8, S, (long long)B * N_c, d_I, s),
            "fp4_to_e4m3 launch");
        if (st != CSA_OK) return st;
        keys = x8;
        ksc = S;
    }
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t elem = fp8 ? 1 : 2;
    const uint32_t box_inner = 128 / elem;
    CUtensorMap tq, tk;
    csa_status_t st = make_map(&tq, q_idx, dt, (uint64_t)d_I, (uint64_t)B * n_q * H_I, (uint64_t)d_I * elem, box_inner,
                               (uint32_t)indexer_box_rows(T));
    if (st != CSA_OK) return st;
    if (kfp4)   // packed rows of d_I / 2 bytes, copied unswizzled for the converter warps
        st = make_map(&tk, keys, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)d_I / 2, (uint64_t)B * N_c, (uint64_t)d_I / 2,
                      (uint32_t)d_I / 2, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        st = make_map(&tk, keys, dt, (uint64_t)d_I, (uint64_t)B * N_c, (uint64_t)d_I * elem, box_inner, 128);
    if (st != CSA_OK) return st;
    return cuda_status(launch_indexer_tc(fp8, T, tq, tk, q_scale, head_w, relu, ksc, scores, sbf16, B, n_q, i_start,
                                         n_q_rows,
                                         q_pos0, m, N_c, num_sms(), wmax, wmax_ld, kfp4, s, zero_words, n_zero),
                       "indexer_tc launch");
}

// The fused route of csa_index_topk: tensor-core scores of decode groups
// (fewer than four queries per sequence in the chunk) over rows longer than
// one top-k CTA's capacity; the indexer also emits the rows' warp maxima, from
// which the top-k takes its collection threshold.
bool fused_index_topk(csa_dtype_t q_dtype, int n_q_rows, int N_c, int k)
{
    return q_dtype != CSA_F32 && indexer_group_tokens(n_q_rows) == 1 && topk_long_rows(N_c, k);
}

}  // namespace

namespace csa {
// Sets the thread's last-error message for entry points defined in other files.
csa_status_t report(csa_status_t st, const char* msg) { return fail(st, "%s", msg); }

// Self-test of the bounded waits: warp 0 waits on an mbarrier that nothing
// completes and gives up after limit_ns (flagging STATUS_TIMEOUT and the CTA's
// abort flag); warp 1 waits on another such barrier under the default limit
// and must stop as soon as the abort flag rises.  No copy, MMA or tensor
// memory is involved, so nothing is in flight when the waits end.
__global__ void wait_selftest_kernel(uint64_t limit_ns, unsigned* stopped_by_abort)
{
    __shared__ uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        if (warp == 0) {
            mbar_wait_for(&bars[0], 0, &abort_flag, limit_ns);
        } else {
            const uint64_t t0 = globaltimer_ns();
            const bool ok = mbar_wait(&bars[1], 0, &abort_flag);
            // stopped by the abort flag, well before its own 2 s limit
            if (!ok && globaltimer_ns() - t0 < WAIT_LIMIT_NS / 2) atomicOr(stopped_by_abort, 1u);
        }
    }
    __syncthreads();
}
}  // namespace csa

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
static csa_status_t check_attn(int B, int n_q, int H, int H_kv, int d, long long N_kv, float scale, const void* q,
                               const void* k, const void* v, csa_dtype_t dtype, const void* out, const float* lse)
{
    if (B < 0 || n_q < 0 || N_kv < 0) return fail(CSA_ERR_INVALID_ARG, "bad sizes");
    if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CSA_ERR_INVALID_ARG, "scale must be positive and finite");
    if (dtype != CSA_F32 && dtype != CSA_BF16) return fail(CSA_ERR_UNSUPPORTED, "attention dtype must be F32 or BF16");
    if (H_kv < 1 || H < H_kv || H % H_kv) return fail(CSA_ERR_INVALID_ARG, "H_kv must divide H (H=%d, H_kv=%d)", H, H_kv);
    if (H_kv == 1 && !attn_simt_supported(H, d))
        return fail(CSA_ERR_UNSUPPORTED, "attention needs H in {8,16,32,64,128}, d in {64,128}");
    const int G = H / H_kv;
    if (H_kv > 1 && ((G & (G - 1)) || G > 128 || (d != 64 && d != 128)))
        return fail(CSA_ERR_UNSUPPORTED, "attention needs H / H_kv a power of two <= 128 and d in {64,128}");
    if ((long long)B * n_q == 0) return CSA_OK;
    if (!q || !out || (N_kv > 0 && (!k || !v))) return fail(CSA_ERR_INVALID_ARG, "NULL tensor");
    if (!aligned16(q) || !aligned16(out) || (k && !aligned16(k)) || (v && !aligned16(v)) || (lse && !aligned16(lse)))
        return fail(CSA_ERR_ALIGNMENT, "attention pointer not 16-byte aligned");
    return CSA_OK;
}

static csa_status_t run_attn_tc(int mode, int B, int n_q, int64_t q_pos0, int m, long long window, long long N_kv,
                               int H, int d, int k, float scale, const void* q, const void* kp, const void* vp,
                               const int32_t* topk, void* out, float* lse, SplitPlan sp, void* ws, cudaStream_t s)
{
    CUtensorMap tq, tk, tv;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    csa_status_t st = make_map(&tq, q, bf, (uint64_t)d, (uint64_t)B * n_q * H, (uint64_t)d * 2, 64,
                               (uint32_t)attn_tc_q_box_rows(mode, H));
    if (st != CSA_OK) return st;
    const uint32_t kv_box = mode == 0 ? 1 : 128;     // row gathers vs 128-key tiles
    st = make_map(&tk, kp, bf, (uint64_t)d, (uint64_t)B * N_kv, (uint64_t)d * 2, 64, kv_box);
    if (st != CSA_OK) return st;
    st = make_map(&tv, vp, bf, (uint64_t)d, (uint64_t)B * N_kv, (uint64_t)d * 2, 64, kv_box);
    if (st != CSA_OK) return st;
    AttnTcParams p{};
    p.topk = topk;
    p.k_rows = reinterpret_cast<const __nv_bfloat16*>(kp);
    p.v_rows = reinterpret_cast<const __nv_bfloat16*>(vp);
    p.out = reinterpret_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.q_pos0 = q_pos0;
    p.window = window;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.B = B;
    p.n_q = n_q;
    p.N_kv = (int)N_kv;
    p.k = k;
    p.m = m;
    p.H = H;
    p.T = attn_tc_tokens_per_cta(mode, H);
    p.n_splits = sp.n;
    p.split_len = sp.len;
    if (sp.n > 1) {
        p.part_o = reinterpret_cast<float*>(ws);
        p.part_ml = p.part_o + (size_t)sp.n * B * n_q * H * d;
    }
    return cuda_status(launch_attn_tc(mode, tq, tk, tv, p, s), "attention (tcgen05) launch");
}

template <typename TIO>
static csa_status_t run_attn(int mode, int B, int n_q, int64_t q_pos0, int m, long long window, long long N_kv, int H,
                             int H_kv, int d, int k, float scale, const void* q, const void* kp, const void* vp,
                             const int32_t* topk, void* out, float* lse, SplitPlan sp, void* ws, cudaStream_t s)
{
    if constexpr (std::is_same<TIO, __nv_bfloat16>::value) {
        // the tensor-core kernel (one shared KV head) stages at most 4096
        // selected entries per CTA
        if (H_kv == 1 && attn_tc_supported(H, d) && N_kv > 0 && (mode != 0 || k <= 4096)) {
            // TMA row coordinates are 32-bit
            if ((long long)B * n_q * H + 128 > INT32_MAX || (long long)B * N_kv + 128 > INT32_MAX)
                return fail(CSA_ERR_UNSUPPORTED, "attention tensors exceed 2^31 rows");
            return run_attn_tc(mode, B, n_q, q_pos0, m, window, N_kv, H, d, k, scale, q, kp, vp, topk, out, lse, sp,
                               ws, s);
        }
    }
    AttnArgsT<TIO> a{};
    a.q = reinterpret_cast<const TIO*>(q);
    a.k_ptr = reinterpret_cast<const TIO*>(kp);
    a.v_ptr = reinterpret_cast<const TIO*>(vp);
    a.out = reinterpret_cast<TIO*>(out);
    a.lse = lse;
    a.topk = topk;
    a.q_pos0 = q_pos0;
    a.window = window;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.mode = mode;
    a.B = B;
    a.n_q = n_q;
    a.N_kv = (int)N_kv;
    a.k = k;
    a.m = m;
    a.n_splits = sp.n;
    a.H_kv = H_kv;
    a.H_tot = H;
    a.G = H / H_kv;
    if (sp.n > 1) {
        a.part_o = reinterpret_cast<float*>(ws);
        a.part_ml = a.part_o + (size_t)sp.n * B * n_q * H * d;
    }
    return cuda_status(launch_attn_simt<TIO>(a, H / H_kv, d, s), "attention launch");
}

static size_t sparse_ws(int B, int n_q, int H, int d, int k)
{
    const SplitPlan sp = attn_split_plan(n_q, k);
    if (sp.n <= 1) return 0;
    return (size_t)sp.n * B * n_q * H * (d + 2) * sizeof(float);
}

static csa_status_t check_index_args(int B, int n_q, int64_t q_pos0, int m, int N_c, int H_I, int d_I,
                                     const void* q_idx, csa_dtype_t q_dtype, const float* q_scale, const void* k_idx,
                                     csa_dtype_t k_dtype, const void* k_scale, const float* head_w = nullptr)
{
    if (head_w && !aligned16(head_w)) return fail(CSA_ERR_ALIGNMENT, "head_weight not 16-byte aligned");
    if (B < 0 || n_q < 0 || m < 1 || N_c < 0 || H_I < 1 || d_I < 1 || q_pos0 < 0)
        return fail(CSA_ERR_INVALID_ARG, "bad sizes");
    csa_status_t st = check_index_dtypes(q_dtype, k_dtype, H_I, d_I);
    if (st != CSA_OK) return st;
    if ((long long)B * n_q * N_c == 0) return CSA_OK;
    if (!q_idx || !k_idx) return fail(CSA_ERR_INVALID_ARG, "NULL q or k");
    if (!aligned16(q_idx) || !aligned16(k_idx) || (q_scale && !aligned16(q_scale)) || (k_scale && !aligned16(k_scale)))
        return fail(CSA_ERR_ALIGNMENT, "indexer pointer not 16-byte aligned");
    if (q_dtype == CSA_E4M3 && !q_scale) return fail(CSA_ERR_INVALID_ARG, "E4M3 queries need q_scale");
    if ((k_dtype == CSA_E4M3 || k_dtype == CSA_E2M1) && !k_scale)
        return fail(CSA_ERR_INVALID_ARG, "quantised keys need k_scale");
    if (k_dtype == CSA_E2M1 && d_I % 32) return fail(CSA_ERR_INVALID_ARG, "E2M1 keys need d_I % 32 == 0");
    return CSA_OK;
}

static csa_status_t check_score_dtype(csa_dtype_t t)
{
    if (t != CSA_F32 && t != CSA_BF16) return fail(CSA_ERR_UNSUPPORTED, "scores must be F32 or BF16 (got %d)", (int)t);
    return CSA_OK;
}

static csa_status_t check_topk(int N_c, int k)
{
    if (!topk_supported(N_c, k)) return fail(CSA_ERR_UNSUPPORTED, "top-k needs 1 <= k <= 4096, N_c <= 524288 (k=%d, N_c=%d)", k, N_c);
    return CSA_OK;
}

extern "C" {

const char* csa_last_error(void) { return g_msg; }

csa_status_t csa_wait_selftest(uint32_t limit_us, uint32_t* aborted, csa_stream_t stream)
{
    if (limit_us < 1 || limit_us > 2000000u) return fail(CSA_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
    if (!aborted || !aligned16(aborted)) return fail(CSA_ERR_ALIGNMENT, "aborted NULL or not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(aborted, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_status(e, "clear aborted flag");
    wait_selftest_kernel<<<1, 64, 0, s>>>((uint64_t)limit_us * 1000ull, reinterpret_cast<unsigned*>(aborted));
    return cuda_status(cudaGetLastError(), "wait self-test launch");
}

csa_status_t csa_device_status(csa_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e, "cudaStreamSynchronize");
    unsigned v = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&v, csa::g_status, sizeof(v));
    if (e != cudaSuccess) return cuda_status(e, "read status word");
    if (v) {
        e = cudaMemcpyToSymbol(csa::g_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_status(e, "clear status word");
    }
    if (v & STATUS_TIMEOUT) return fail(CSA_ERR_TIMEOUT, "a device wait exceeded its time limit");
    if (v & STATUS_BOUNDS) return fail(CSA_ERR_DEVICE, "a device-side bounds check failed");
    return CSA_OK;
}

// Argument checks shared by the compression entry points.
static csa_status_t check_compress_streams(int n_streams, const void* const* x, const csa_dtype_t* x_dtype,
                                           const int* dim, void* const* out, const csa_dtype_t* out_dtype,
                                           void* const* out_scale)
{
    for (int s = 0; s < n_streams; ++s) {
        const int d = dim[s];
        const bool pow2 = d >= 8 && d <= 256 && (d & (d - 1)) == 0;
        if (!pow2) return fail(CSA_ERR_UNSUPPORTED, "stream %d: dim %d not a power of two in [8, 256]", s, d);
        if (x_dtype[s] != CSA_F32 && x_dtype[s] != CSA_BF16)
            return fail(CSA_ERR_INVALID_ARG, "stream %d: input dtype must be F32 or BF16", s);
        if (!x[s] || !out[s]) return fail(CSA_ERR_INVALID_ARG, "stream %d: NULL pointer", s);
        if (!aligned16(x[s]) || !aligned16(out[s])) return fail(CSA_ERR_ALIGNMENT, "stream %d: pointer not 16-byte aligned", s);
        const csa_dtype_t od = out_dtype[s];
        if (od == CSA_E4M3 || od == CSA_E2M1) {
            if (!out_scale || !out_scale[s]) return fail(CSA_ERR_INVALID_ARG, "stream %d: quantised output needs out_scale", s);
            if (od == CSA_E4M3 && !aligned16(out_scale[s])) return fail(CSA_ERR_ALIGNMENT, "stream %d: scale not aligned", s);
            if (od == CSA_E2M1 && d < 32) return fail(CSA_ERR_UNSUPPORTED, "stream %d: E2M1 needs dim >= 32", s);
        } else if (od != CSA_F32 && od != CSA_BF16) {
            return fail(CSA_ERR_INVALID_ARG, "stream %d: bad output dtype", s);
        }
    }
    return CSA_OK;
}

static int out_kind_of(csa_dtype_t od) { return od == CSA_F32 ? 0 : od == CSA_BF16 ? 1 : od == CSA_E4M3 ? 2 : 3; }

csa_status_t csa_compress(int B, int n, int m, const float* logits, int n_streams, const void* const* x,
                          const csa_dtype_t* x_dtype, const int* dim, void* const* out, const csa_dtype_t* out_dtype,
                          void* const* out_scale, csa_stream_t stream)
{
    if (B < 0 || n < 0 || m < 1) return fail(CSA_ERR_INVALID_ARG, "bad sizes B=%d n=%d m=%d", B, n, m);
    if (n_streams < 1 || n_streams > 4 || !x || !x_dtype || !dim || !out || !out_dtype)
        return fail(CSA_ERR_INVALID_ARG, "bad stream arrays (n_streams=%d)", n_streams);
    const int Nc = n / m;
    if ((long long)B * Nc == 0) return CSA_OK;
    if (!logits) return fail(CSA_ERR_INVALID_ARG, "logits is NULL");
    if (!aligned16(logits)) return fail(CSA_ERR_ALIGNMENT, "logits not 16-byte aligned");
    csa_status_t cst = check_compress_streams(n_streams, x, x_dtype, dim, out, out_dtype, out_scale);
    if (cst != CSA_OK) return cst;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int kinds[4];
    bool bf16_in[4];
    for (int s = 0; s < n_streams; ++s) {
        kinds[s] = out_kind_of(out_dtype[s]);
        bf16_in[s] = x_dtype[s] == CSA_BF16;
    }
    if (compress_tiles_supported(n, m, n_streams, dim, bf16_in)) {
        cudaError_t e = launch_compress_tiles(B, n, m, n_streams, logits, x, bf16_in, dim, out, kinds, out_scale,
                                              num_sms(), st);
        if (e != cudaSuccess) return cuda_status(e, "compress launch");
        return CSA_OK;
    }
    for (int s = 0; s < n_streams; ++s) {
        cudaError_t e = launch_compress(B, n, m, dim[s], logits, x[s], bf16_in[s], out[s], kinds[s],
                                        out_scale ? out_scale[s] : nullptr, num_sms(), st);
        if (e != cudaSuccess) return cuda_status(e, "compress launch");
    }
    return CSA_OK;
}

csa_status_t csa_compress_per_channel(int B, int n, int m, int n_streams, const float* const* logits,
                                      const void* const* x, const csa_dtype_t* x_dtype, const int* dim,
                                      void* const* out, const csa_dtype_t* out_dtype, void* const* out_scale,
                                      csa_stream_t stream)
{
    if (B < 0 || n < 0 || m < 1) return fail(CSA_ERR_INVALID_ARG, "bad sizes B=%d n=%d m=%d", B, n, m);
    if (n_streams < 1 || n_streams > 4 || !logits || !x || !x_dtype || !dim || !out || !out_dtype)
        return fail(CSA_ERR_INVALID_ARG, "bad stream arrays (n_streams=%d)", n_streams);
    if ((long long)B * (n / m) == 0) return CSA_OK;
    for (int s = 0; s < n_streams; ++s) {
        if (!logits[s]) return fail(CSA_ERR_INVALID_ARG, "stream %d: logits NULL", s);
        if (!aligned16(logits[s])) return fail(CSA_ERR_ALIGNMENT, "stream %d: logits not 16-byte aligned", s);
    }
    csa_status_t cst = check_compress_streams(n_streams, x, x_dtype, dim, out, out_dtype, out_scale);
    if (cst != CSA_OK) return cst;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int s = 0; s < n_streams; ++s) {
        cudaError_t e = launch_compress_per_channel(B, n, m, dim[s], logits[s], x[s], x_dtype[s] == CSA_BF16, out[s],
                                                    out_kind_of(out_dtype[s]), out_scale ? out_scale[s] : nullptr, st);
        if (e != cudaSuccess) return cuda_status(e, "compress (per channel) launch");
    }
    return CSA_OK;
}

csa_status_t csa_decode_append(int B, int m, int d, int d_I, int64_t N_cap, const float* logit_new,
                               const void* k_new, const void* v_new, const void* ik_new, csa_dtype_t x_dtype,
                               float* stage_logits, void* stage_k, void* stage_v, void* stage_ik, int64_t* lens,
                               void* k_c, void* v_c, csa_dtype_t kv_dtype, void* ik_c, csa_dtype_t ik_dtype,
                               void* ik_scale, csa_stream_t stream)
{
    if (B < 0 || m < 1 || N_cap < 0) return fail(CSA_ERR_INVALID_ARG, "bad sizes B=%d m=%d", B, m);
    if (m > DECODE_MAX_M) return fail(CSA_ERR_UNSUPPORTED, "decode append needs m <= %d", DECODE_MAX_M);
    if (d < 1 || d > DECODE_MAX_DIM || d_I < 2 || d_I > DECODE_MAX_DIM || (d_I & 1))
        return fail(CSA_ERR_UNSUPPORTED, "decode append needs d, d_I <= %d (d_I even)", DECODE_MAX_DIM);
    if (x_dtype != CSA_F32 && x_dtype != CSA_BF16) return fail(CSA_ERR_INVALID_ARG, "new tokens must be F32 or BF16");
    if (kv_dtype != CSA_F32 && kv_dtype != CSA_BF16) return fail(CSA_ERR_INVALID_ARG, "K/V caches must be F32 or BF16");
    if (ik_dtype == CSA_E2M1 && d_I % 32) return fail(CSA_ERR_UNSUPPORTED, "E2M1 indexer keys need d_I % 32 == 0");
    if (B == 0) return CSA_OK;
    const void* ptrs[] = {logit_new, k_new, v_new, ik_new, stage_logits, stage_k, stage_v, stage_ik, lens, k_c, v_c, ik_c};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return fail(CSA_ERR_ALIGNMENT, "decode append: pointer NULL or not 16-byte aligned");
    if ((ik_dtype == CSA_E4M3 || ik_dtype == CSA_E2M1) && (!ik_scale || !aligned16(ik_scale)))
        return fail(CSA_ERR_INVALID_ARG, "quantised indexer keys need an aligned ik_scale");
    DecodeAppendArgs a{};
    a.B = B; a.m = m; a.d = d; a.d_I = d_I; a.N_cap = N_cap;
    a.logit_new = logit_new; a.k_new = k_new; a.v_new = v_new; a.ik_new = ik_new;
    a.st_logit = stage_logits; a.st_k = stage_k; a.st_v = stage_v; a.st_ik = stage_ik;
    a.lens = reinterpret_cast<long long*>(lens);
    a.k_c = k_c; a.v_c = v_c; a.kv_kind = kv_dtype == CSA_BF16 ? 1 : 0;
    a.ik_c = ik_c; a.ik_scale = ik_scale;
    a.ik_kind = ik_dtype == CSA_F32 ? 0 : ik_dtype == CSA_BF16 ? 1 : ik_dtype == CSA_E4M3 ? 2 : 3;
    return cuda_status(launch_decode_append(a, x_dtype == CSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                       "decode append launch");
}

size_t csa_index_scores_workspace_size(int B, int N_c, int d_I, csa_dtype_t k_dtype)
{
    if (B < 0 || N_c < 0 || d_I < 0) return 0;
    return scores_ws_bytes(B, N_c, d_I, k_dtype);
}


csa_status_t csa_index_scores(int B, int n_q, int64_t q_pos0, int m, int N_c, int H_I, int d_I, const void* q_idx,
                              csa_dtype_t q_dtype, const float* q_scale, const void* k_idx, csa_dtype_t k_dtype,
                              const void* k_scale, const float* head_weight, int relu, void* scores,
                              csa_dtype_t score_dtype, void* workspace, size_t workspace_bytes, csa_stream_t stream)
{
    csa_status_t st = check_index_args(B, n_q, q_pos0, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                                       head_weight);
    if (st != CSA_OK) return st;
    st = check_score_dtype(score_dtype);
    if (st != CSA_OK) return st;
    if ((long long)B * n_q * N_c == 0) return CSA_OK;
    if (!scores || !aligned16(scores)) return fail(CSA_ERR_ALIGNMENT, "scores NULL or not aligned");
    const size_t need = scores_ws_bytes(B, N_c, d_I, k_dtype);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return fail(CSA_ERR_WORKSPACE, "workspace needs %zu bytes", need);
    return run_scores(B, n_q, 0, n_q, q_pos0, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                      head_weight, relu != 0, scores, score_dtype == CSA_BF16, workspace,
                      reinterpret_cast<cudaStream_t>(stream));
}

size_t csa_topk_select_workspace_size(int B, int n_q, int N_c, int k)
{
    if (B < 0 || n_q < 0 || N_c < 0 || k < 1) return 0;
    return topk_workspace_bytes((long long)B * n_q, N_c, k);
}


csa_status_t csa_topk_select(int B, int n_q, int64_t q_pos0, int m, int N_c, int k, const void* scores,
                             csa_dtype_t score_dtype, int32_t* topk, void* workspace, size_t workspace_bytes,
                             csa_stream_t stream)
{
    if (B < 0 || n_q < 0 || m < 1 || N_c < 0 || q_pos0 < 0) return fail(CSA_ERR_INVALID_ARG, "bad sizes");
    csa_status_t st = check_topk(N_c, k);
    if (st != CSA_OK) return st;
    st = check_score_dtype(score_dtype);
    if (st != CSA_OK) return st;
    const long long rows = (long long)B * n_q;
    if (rows == 0) return CSA_OK;
    if (!topk_rows_ok(rows, N_c, k)) return fail(CSA_ERR_UNSUPPORTED, "top-k over %lld rows exceeds the grid limit", rows);
    if (!topk || !aligned16(topk) || (N_c > 0 && (!scores || !aligned16(scores))))
        return fail(CSA_ERR_ALIGNMENT, "scores/topk NULL or not aligned");
    const size_t need = topk_workspace_bytes(rows, N_c, k);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return fail(CSA_ERR_WORKSPACE, "workspace needs %zu bytes", need);
    return cuda_status(launch_topk(scores, score_dtype == CSA_BF16, N_c, B, n_q, q_pos0, m, N_c, k, topk, n_q, workspace,
                                   reinterpret_cast<cudaStream_t>(stream)),
                       "topk launch");
}

size_t csa_index_topk_workspace_size(int B, int n_q, int N_c, int H_I, int d_I, int k, csa_dtype_t k_dtype,
                                     csa_dtype_t score_dtype)
{
    if (B < 0 || n_q < 0 || N_c < 0 || k < 1) return 0;
    const size_t esz = score_dtype == CSA_BF16 ? 2 : 4;
    const int rows = index_chunk_rows(B, n_q, N_c, esz);
    return align_up((size_t)B * rows * N_c * esz, 256) + scores_ws_bytes(B, N_c, d_I, k_dtype) +
           topk_workspace_bytes((long long)B * rows, N_c, k) +
           (topk_long_rows(N_c, k) ? topk_wmax_bytes((long long)B * rows, N_c) : 0);
}

// csa_index_topk and csa_index_topk_varlen: positions are q_pos0 for every
// sequence, or (lens non-null) lens[b] - n_q for sequence b.
static csa_status_t index_topk_impl(int B, int n_q, int64_t q_pos0, const int64_t* lens, int m, int N_c, int H_I,
                                    int d_I, int k, const void* q_idx, csa_dtype_t q_dtype, const float* q_scale,
                                    const void* k_idx, csa_dtype_t k_dtype, const void* k_scale,
                                    const float* head_weight, int relu, csa_dtype_t score_dtype, int32_t* topk,
                                    void* workspace, size_t workspace_bytes, csa_stream_t stream)
{
    csa_status_t st = check_index_args(B, n_q, q_pos0, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                                       head_weight);
    if (st != CSA_OK) return st;
    st = check_topk(N_c, k);
    if (st != CSA_OK) return st;
    st = check_score_dtype(score_dtype);
    if (st != CSA_OK) return st;
    const bool sbf16 = score_dtype == CSA_BF16;
    const size_t esz = sbf16 ? 2 : 4;
    if ((long long)B * n_q == 0) return CSA_OK;
    if (!topk_rows_ok((long long)B * index_chunk_rows(B, n_q, N_c, esz), N_c, k))
        return fail(CSA_ERR_UNSUPPORTED, "top-k over %d sequences exceeds the grid limit", B);
    if (!topk || !aligned16(topk)) return fail(CSA_ERR_ALIGNMENT, "topk NULL or not aligned");
    const size_t need = csa_index_topk_workspace_size(B, n_q, N_c, H_I, d_I, k, k_dtype, score_dtype);
    if (!workspace || workspace_bytes < need || !aligned16(workspace))
        return fail(CSA_ERR_WORKSPACE, "workspace needs %zu bytes", need);
    if (lens && !aligned16(lens)) return fail(CSA_ERR_ALIGNMENT, "lens not 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the scores' positions (the indexer adds the chunk's first row itself)
    const QPos qp = lens ? QPos(reinterpret_cast<const long long*>(lens), -(long long)n_q) : QPos(q_pos0);
    const int rows = index_chunk_rows(B, n_q, N_c, esz);
    uint8_t* w = reinterpret_cast<uint8_t*>(workspace);
    void* scores = w;
    uint8_t* w_scores_ws = w + align_up((size_t)B * rows * N_c * esz, 256);
    uint8_t* w_topk = w_scores_ws + scores_ws_bytes(B, N_c, d_I, k_dtype);
    uint32_t* w_wmax = reinterpret_cast<uint32_t*>(w_topk + topk_workspace_bytes((long long)B * rows, N_c, k));
    for (int i0 = 0; i0 < n_q; i0 += rows) {
        const int nr = std::min(rows, n_q - i0);
        if (N_c > 0 && fused_index_topk(q_dtype, nr, N_c, k)) {
            // scores plus the rows' warp maxima in one kernel, which also
            // clears the top-k's row counters, then the top-k with its
            // collection threshold taken from the maxima
            const int ld = topk_wmax_ld(N_c);
            st = run_scores(B, n_q, i0, nr, qp, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                            head_weight, relu != 0, scores, sbf16, w_scores_ws, s, w_wmax, ld,
                            topk_row_counters(w_topk), B * nr);
            if (st != CSA_OK) return st;
            st = cuda_status(launch_topk(scores, sbf16, N_c, B, nr, qp.shifted(i0), m, N_c, k, topk + (size_t)i0 * k, n_q,
                                         w_topk, s, w_wmax, ld, true),
                             "topk launch");
            if (st != CSA_OK) return st;
            continue;
        }
        if (N_c > 0) {
            st = run_scores(B, n_q, i0, nr, qp, m, N_c, H_I, d_I, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                            head_weight, relu != 0, scores, sbf16, w_scores_ws, s);
            if (st != CSA_OK) return st;
        }
        st = cuda_status(launch_topk(scores, sbf16, N_c, B, nr, qp.shifted(i0), m, N_c, k, topk + (size_t)i0 * k, n_q, w_topk, s),
                         "topk launch");
        if (st != CSA_OK) return st;
    }
    return CSA_OK;
}

csa_status_t csa_index_topk(int B, int n_q, int64_t q_pos0, int m, int N_c, int H_I, int d_I, int k,
                            const void* q_idx, csa_dtype_t q_dtype, const float* q_scale, const void* k_idx,
                            csa_dtype_t k_dtype, const void* k_scale, const float* head_weight, int relu,
                            csa_dtype_t score_dtype, int32_t* topk, void* workspace, size_t workspace_bytes,
                            csa_stream_t stream)
{
    return index_topk_impl(B, n_q, q_pos0, nullptr, m, N_c, H_I, d_I, k, q_idx, q_dtype, q_scale, k_idx, k_dtype,
                           k_scale, head_weight, relu, score_dtype, topk, workspace, workspace_bytes, stream);
}

csa_status_t csa_index_topk_varlen(int B, int n_q, const int64_t* lens, int m, int N_c, int H_I, int d_I, int k,
                                   const void* q_idx, csa_dtype_t q_dtype, const float* q_scale, const void* k_idx,
                                   csa_dtype_t k_dtype, const void* k_scale, const float* head_weight, int relu,
                                   csa_dtype_t score_dtype, int32_t* topk, void* workspace, size_t workspace_bytes,
                                   csa_stream_t stream)
{
    if (!lens && (long long)B * n_q > 0) return fail(CSA_ERR_INVALID_ARG, "lens is NULL");
    return index_topk_impl(B, n_q, 0, lens, m, N_c, H_I, d_I, k, q_idx, q_dtype, q_scale, k_idx, k_dtype, k_scale,
                           head_weight, relu, score_dtype, topk, workspace, workspace_bytes, stream);
}

size_t csa_sparse_attn_workspace_size(int B, int n_q, int H, int d, int k)
{
    if (B < 0 || n_q < 0 || H < 1 || d < 1 || k < 1) return 0;
    return sparse_ws(B, n_q, H, d, k);
}

csa_status_t csa_sparse_attn(int B, int n_q, int H, int H_kv, int d, int N_c, int k, float scale, const void* q,
                             const void* k_c, const void* v_c, csa_dtype_t dtype, const int32_t* topk, void* out,
                             float* lse, void* workspace, size_t workspace_bytes, csa_stream_t stream)
{
    csa_status_t st = check_attn(B, n_q, H, H_kv, d, N_c, scale, q, k_c, v_c, dtype, out, lse);
    if (st != CSA_OK) return st;
    if (k < 1) return fail(CSA_ERR_INVALID_ARG, "k must be >= 1");
    if ((long long)B * n_q == 0) return CSA_OK;
    if (!topk || !aligned16(topk)) return fail(CSA_ERR_ALIGNMENT, "topk NULL or not aligned");
    const SplitPlan splits = attn_split_plan(n_q, k);
    const size_t need = sparse_ws(B, n_q, H, d, k);
    if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return fail(CSA_ERR_WORKSPACE, "workspace needs %zu bytes", need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == CSA_BF16)
        return run_attn<__nv_bfloat16>(0, B, n_q, 0, 1, 0, N_c, H, H_kv, d, k, scale, q, k_c, v_c, topk, out, lse, splits,
                                       workspace, s);
    return run_attn<float>(0, B, n_q, 0, 1, 0, N_c, H, H_kv, d, k, scale, q, k_c, v_c, topk, out, lse, splits, workspace,
                           s);
}

csa_status_t hca_attn(int B, int n_q, int64_t q_pos0, int m, int N_c, int H, int H_kv, int d, float scale,
                      const void* q, const void* k_c, const void* v_c, csa_dtype_t dtype, void* out, float* lse,
                      csa_stream_t stream)
{
    if (m < 1 || q_pos0 < 0) return fail(CSA_ERR_INVALID_ARG, "bad m / q_pos0");
    csa_status_t st = check_attn(B, n_q, H, H_kv, d, N_c, scale, q, k_c, v_c, dtype, out, lse);
    if (st != CSA_OK) return st;
    if ((long long)B * n_q == 0) return CSA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == CSA_BF16)
        return run_attn<__nv_bfloat16>(1, B, n_q, q_pos0, m, 0, N_c, H, H_kv, d, 0, scale, q, k_c, v_c, nullptr, out,
                                       lse, SplitPlan{1, 1 << 30}, nullptr, s);
    return run_attn<float>(1, B, n_q, q_pos0, m, 0, N_c, H, H_kv, d, 0, scale, q, k_c, v_c, nullptr, out, lse,
                           SplitPlan{1, 1 << 30}, nullptr, s);
}

csa_status_t swa_attn(int B, int n_q, int64_t q_pos0, int n_kv, int window, int H, int H_kv, int d, float scale,
                      const void* q, const void* k, const void* v, csa_dtype_t dtype, void* out, float* lse,
                      csa_stream_t stream)
{
    if (window < 1 || q_pos0 < 0) return fail(CSA_ERR_INVALID_ARG, "bad window / q_pos0");
    csa_status_t st = check_attn(B, n_q, H, H_kv, d, n_kv, scale, q, k, v, dtype, out, lse);
    if (st != CSA_OK) return st;
    if ((long long)B * n_q == 0) return CSA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == CSA_BF16)
        return run_attn<__nv_bfloat16>(2, B, n_q, q_pos0, 1, window, n_kv, H, H_kv, d, 0, scale, q, k, v, nullptr, out,
                                       lse, SplitPlan{1, 1 << 30}, nullptr, s);
    return run_attn<float>(2, B, n_q, q_pos0, 1, window, n_kv, H, H_kv, d, 0, scale, q, k, v, nullptr, out, lse,
                           SplitPlan{1, 1 << 30}, nullptr, s);
}

}  // extern "C"
