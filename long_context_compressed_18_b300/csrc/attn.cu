// Attention of H query heads over one shared KV head (or, in the GQA / MHA
// variant readings, over H_kv KV heads, query head h reading KV head
// h / (H / H_kv)), for the three key sets of the hybrid stack ("DeepSeek V4
// 技术解读"):
//   mode 0  CSA core attention over the top-k selected entries (§2.1),
//   mode 1  HCA dense attention over all closed compressed blocks (§2.2),
//   mode 2  sliding-window attention over raw tokens (§2.3).
//
// CUDA-core kernel.  One CTA handles one query token and one KV head (the
// query heads that share it; at least 8 rows, idle ones never stored) over one
// contiguous slice of its key set; keys are staged in shared memory in tiles
// of 32 (gathered by index for mode 0), scores and an online softmax (base-2,
// fp32) run in registers, and P.V accumulates per thread over a slice of the
// head dim.  When the key set is split across CTAs (short-query decode), each
// CTA writes an unnormalised partial (o, m, l) and a combine kernel merges
// them in split order, so results are deterministic.
#include "common.cuh"
#include "kernels.h"
#include "attn_merge.cuh"

namespace csa {

constexpr int ATT_THREADS = 256;
constexpr int ATT_KT = 32;   // keys per tile

template <typename TIO, int H, int D>
__global__ void __launch_bounds__(ATT_THREADS) attn_simt_kernel(AttnArgsT<TIO> a)
{
    grid_dep_entry();
    constexpr int TPH = ATT_THREADS / H;   // threads per head
    constexpr int KPT = ATT_KT / TPH;      // keys per thread per tile
    constexpr int CPT = D / TPH;           // output channels per thread
    constexpr int QLD = D + 4;             // padded row pitch (floats)
    static_assert(KPT >= 1 && CPT >= 1, "shape");

    extern __shared__ __align__(16) float sm[];
    float* Qs = sm;                        // [H][QLD]
    float* Ks = Qs + H * QLD;              // [KT][QLD]
    float* Vs = Ks + ATT_KT * QLD;         // [KT][D]
    int* kvalid = reinterpret_cast<int*>(Vs + ATT_KT * D);
    int* kidx = kvalid + ATT_KT;

    const int tid = threadIdx.x;
    const int h = tid / TPH, tq = tid % TPH;
    const int lane = tid & 31;
    const unsigned gmask = (TPH >= 32) ? 0xFFFFFFFFu : (((1u << TPH) - 1u) << (lane & ~(TPH - 1)));
    const int b = blockIdx.y;
    const int i = blockIdx.x / a.n_splits, split = blockIdx.x % a.n_splits;
    const long long row = (long long)b * a.n_q + i;
    const long long t = a.q_pos0 + i;
    const int kvh = blockIdx.z;                    // this CTA's KV head
    const int HT = a.H_tot;                        // query heads of a token
    const int h0 = kvh * a.G;                      // its first query head
    const bool h_live = h < a.G;                   // rows past G (when G < H) are idle

    // key-set slice [lo, hi) of this CTA: list positions (mode 0) or key indices
    long long set_lo, set_len;
    if (a.mode == 0) { set_lo = 0; set_len = a.k; }
    else if (a.mode == 1) { long long nv = (t + 1) / a.m; set_lo = 0; set_len = nv < a.N_kv ? nv : a.N_kv; }
    else {
        long long lo = t - a.window + 1; if (lo < 0) lo = 0;
        long long hi = t < a.N_kv - 1 ? t : a.N_kv - 1;
        set_lo = lo; set_len = hi >= lo ? hi - lo + 1 : 0;
    }
    const long long per = (set_len + a.n_splits - 1) / a.n_splits;
    const long long s_lo = set_lo + (long long)split * per;
    const long long s_hi = set_lo + min(set_len, (long long)(split + 1) * per);

    // stage Q (pre-scaled to the base-2 domain); idle rows are zero
    const TIO* qp = a.q + (row * HT + h0) * D;
    for (int x = tid * 8; x < H * D; x += ATT_THREADS * 8) {
        float v[8];
        const int hh = x / D, c = x % D;
        if (hh < a.G) {
            Vec8<TIO>::load(qp + x, v);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) Qs[hh * QLD + c + u] = v[u] * a.scale_log2;
    }

    float o[CPT];
#pragma unroll
    for (int u = 0; u < CPT; ++u) o[u] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    const int32_t* sel = (a.mode == 0) ? a.topk + row * a.k : nullptr;

    for (long long base = s_lo; base < s_hi; base += ATT_KT) {
        __syncthreads();   // previous tile fully consumed (and Q staged on the first pass)
        if (tid < ATT_KT) {
            const long long pos = base + tid;
            int valid = 0;
            long long j = -1;
            if (pos < s_hi) {
                if (a.mode == 0) {
                    j = sel[pos];
                    if (j >= a.N_kv) { flag_status(STATUS_BOUNDS); j = -1; }
                } else {
                    j = pos;
                }
                valid = j >= 0;
            }
            kvalid[tid] = valid;
            kidx[tid] = valid ? (int)j : 0;
        }
        __syncthreads();
        for (int x = tid; x < ATT_KT * (D / 8); x += ATT_THREADS) {
            const int e = x / (D / 8), c = (x % (D / 8)) * 8;
            float kv[8], vv[8];
            if (kvalid[e]) {
                const long long off = (((long long)b * a.N_kv + kidx[e]) * a.H_kv + kvh) * D + c;
                Vec8<TIO>::load(a.k_ptr + off, kv);
                Vec8<TIO>::load(a.v_ptr + off, vv);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) { kv[u] = 0.f; vv[u] = 0.f; }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) { Ks[e * QLD + c + u] = kv[u]; Vs[e * D + c + u] = vv[u]; }
        }
        __syncthreads();

        // scores for this thread's keys e = tq + kk * TPH
        float s[KPT];
#pragma unroll
        for (int kk = 0; kk < KPT; ++kk) s[kk] = 0.f;
        const float* qh = Qs + h * QLD;
#pragma unroll 4
        for (int c = 0; c < D; c += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(qh + c);
#pragma unroll
            for (int kk = 0; kk < KPT; ++kk) {
                const float4 k4 = *reinterpret_cast<const float4*>(Ks + (tq + kk * TPH) * QLD + c);
                s[kk] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, s[kk]))));
            }
        }
        float mt = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < KPT; ++kk) {
            if (!kvalid[tq + kk * TPH]) s[kk] = -INFINITY;
            mt = fmaxf(mt, s[kk]);
        }
#pragma unroll
        for (int off = TPH / 2; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(gmask, mt, off, TPH));
        const float m_new = fmaxf(m_run, mt);
        if (m_new == -INFINITY) continue;   // nothing valid yet (uniform per head group)
        const float alpha = exp2f(m_run - m_new);
        float psum = 0.f;
#pragma unroll
        for (int kk = 0; kk < KPT; ++kk) { s[kk] = exp2f(s[kk] - m_new); psum += s[kk]; }
#pragma unroll
        for (int off = TPH / 2; off > 0; off >>= 1) psum += __shfl_xor_sync(gmask, psum, off, TPH);
        l_run = l_run * alpha + psum;
        m_run = m_new;
#pragma unroll
        for (int u = 0; u < CPT; ++u) o[u] *= alpha;
        const int c0 = tq * CPT;
#pragma unroll
        for (int e = 0; e < ATT_KT; ++e) {
            const float pe = __shfl_sync(gmask, s[e / TPH], (lane & ~(TPH - 1)) + (e % TPH), 32);
            const float* vr = Vs + e * D + c0;
#pragma unroll
            for (int u = 0; u < CPT; ++u) o[u] = fmaf(pe, vr[u], o[u]);
        }
    }

    // finish
    if (a.n_splits == 1) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        float ov[CPT];
#pragma unroll
        for (int u = 0; u < CPT; ++u) ov[u] = o[u] * inv;
        TIO* op = a.out + (row * HT + h0 + h) * D + tq * CPT;
        if (!h_live) return;
        if constexpr (CPT % 8 == 0) {
#pragma unroll
            for (int u = 0; u < CPT; u += 8) {
                float tmp[8];
#pragma unroll
                for (int w = 0; w < 8; ++w) tmp[w] = ov[u + w];
                Vec8<TIO>::store(op + u, tmp);
            }
        } else {
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
                if constexpr (sizeof(TIO) == 4) op[u] = ov[u];
                else op[u] = __float2bfloat16_rn(ov[u]);
            }
        }
        if (a.lse && tq == 0)
            a.lse[row * HT + h0 + h] = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    } else {
        if (!h_live) return;
        const long long prow = ((long long)split * a.B * a.n_q + row) * HT + h0 + h;
        float* po = a.part_o + prow * D + tq * CPT;
#pragma unroll
        for (int u = 0; u < CPT; ++u) po[u] = o[u];
        if (tq == 0) { a.part_ml[2 * prow] = m_run; a.part_ml[2 * prow + 1] = l_run; }
    }
}

// Merge split partials (attn_merge.cuh).  One thread per (row, head, 8 channels).
template <typename TIO>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgsT<TIO> a, int H, int D)
{
    grid_dep_entry();
    const long long n = (long long)a.B * a.n_q * H * (D / 8);
    const long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n) return;
    merge_split_partials(a, H, D, x / (D / 8), (int)(x % (D / 8)) * 8);
}

size_t attn_smem_bytes(int H, int D)
{
    return (size_t)(H * (D + 4) + ATT_KT * (D + 4) + ATT_KT * D) * sizeof(float) + 2 * ATT_KT * sizeof(int);
}

template <typename TIO, int H, int D>
static cudaError_t launch_h(const AttnArgsT<TIO>& a, cudaStream_t s)
{
    auto kern = attn_simt_kernel<TIO, H, D>;
    const size_t smem = attn_smem_bytes(H, D);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    dim3 grid(a.n_q * a.n_splits, a.B, a.H_kv);
    (void)launch_pdl(kern, dim3(grid), dim3(ATT_THREADS), smem, s, a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.n_splits == 1) return e;
    const long long n = (long long)a.B * a.n_q * a.H_tot * (D / 8);
    (void)launch_pdl(attn_combine_kernel<TIO>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, a, a.H_tot, D);
    return cudaGetLastError();
}

cudaError_t launch_attn_combine(const AttnArgsT<__nv_bfloat16>& a, int H, int D, cudaStream_t s)
{
    const long long n = (long long)a.B * a.n_q * H * (D / 8);
    if (n == 0) return cudaSuccess;
    (void)launch_pdl(attn_combine_kernel<__nv_bfloat16>, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, a, H, D);
    return cudaGetLastError();
}

template <typename TIO, int D>
static cudaError_t launch_d(const AttnArgsT<TIO>& a, int H, cudaStream_t s)
{
    // a CTA's rows: the G query heads of one KV head, at least 8
    switch (H < 8 ? 8 : H) {
        case 8: return launch_h<TIO, 8, D>(a, s);
        case 16: return launch_h<TIO, 16, D>(a, s);
        case 32: return launch_h<TIO, 32, D>(a, s);
        case 64: return launch_h<TIO, 64, D>(a, s);
        case 128: return launch_h<TIO, 128, D>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TIO>
cudaError_t launch_attn_simt(const AttnArgsT<TIO>& a_in, int H, int D, cudaStream_t s)
{
    if (a_in.B * a_in.n_q == 0) return cudaSuccess;
    AttnArgsT<TIO> a = a_in;
    if (a.H_tot == 0) {   // one shared KV head
        a.H_kv = 1;
        a.H_tot = H;
        a.G = H;
    }
    if (D == 64) return launch_d<TIO, 64>(a, H, s);
    return launch_d<TIO, 128>(a, H, s);
}

bool attn_simt_supported(int H, int D)
{
    return (H == 8 || H == 16 || H == 32 || H == 64 || H == 128) && (D == 64 || D == 128);
}

template cudaError_t launch_attn_simt<float>(const AttnArgsT<float>&, int, int, cudaStream_t);
template cudaError_t launch_attn_simt<__nv_bfloat16>(const AttnArgsT<__nv_bfloat16>&, int, int, cudaStream_t);

}  // namespace csa
