// KV compression ("DeepSeek V4 技术解读" §2.1 KV Cache 压缩 and §2.2 HCA):
// every block of m raw tokens becomes one entry, the softmax-weighted sum of
// its tokens (one scalar logit per token).  Optional epilogues quantise the
// compressed entry to E4M3 (per-row fp32 scale) or E2M1 (E4M3 scale per 32
// elements) for the Lightning Indexer's FP8 / FP4 key cache.
//
// HBM-bound streaming reduction.  One thread owns 8 consecutive channels of
// one output entry: it issues m 16-byte (bf16) or 2x16-byte (fp32) loads,
// coalesced across the G = d/8 threads of the row, and accumulates in fp32 in
// token order.  The softmax statistics of a block are reduced across the row's
// thread group with shuffles; row / block maxima for the quantisers likewise.
#include "common.cuh"
#include "kernels.h"

namespace csa {

// At most 64 registers a thread, so at least four CTAs (32 warps) share an SM
// and keep enough 16-byte loads in flight for HBM when a block is short (m = 4).
template <typename Tin, int OUT>
__global__ void __launch_bounds__(256, 4) compress_kernel(int B, int n, int m, int Nc, int d,
                                                       const float* __restrict__ logits,
                                                       const Tin* __restrict__ x, void* out,
                                                       void* out_scale)
{
    const int G = d >> 3;  // threads per output row (power of two, <= 32)
    const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long rows = (long long)B * Nc;
    const long long row = gtid / G;
    const int g = (int)(gtid % G);
    const bool live = row < rows;
    const long long r = live ? row : rows - 1;  // dead lanes mirror the last row
    const long long b = r / Nc, j = r % Nc;
    const unsigned lane = threadIdx.x & 31;
    const unsigned gmask = (G == 32) ? 0xFFFFFFFFu : (((1u << G) - 1u) << (lane & ~(unsigned)(G - 1)));

    // softmax statistics of the block's m logits, split across the row group
    const float* lg = logits + b * (long long)n + j * (long long)m;
    float mx = -INFINITY;
    for (int i = g; i < m; i += G) mx = fmaxf(mx, __ldg(lg + i));
    for (int o = G >> 1; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(gmask, mx, o, G));
    float den = 0.f;
    for (int i = g; i < m; i += G) den += expf(__ldg(lg + i) - mx);
    for (int o = G >> 1; o > 0; o >>= 1) den += __shfl_xor_sync(gmask, den, o, G);

    // weighted sum over the block's tokens, in token order
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    const Tin* xp = x + (b * (long long)n + j * (long long)m) * d + 8 * g;
#pragma unroll 4
    for (int i = 0; i < m; ++i) {
        float v[8];
        Vec8<Tin>::load(xp + (long long)i * d, v);
        const float e = expf(__ldg(lg + i) - mx);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = fmaf(e, v[c], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = __fdiv_rn(acc[c], den);

    if constexpr (OUT == 0 || OUT == 1) {
        using Tout = typename std::conditional<OUT == 0, float, __nv_bfloat16>::type;
        if (live) Vec8<Tout>::store(reinterpret_cast<Tout*>(out) + r * d + 8 * g, acc);
    } else if constexpr (OUT == 2) {
        // E4M3 codes with one fp32 scale per row: scale = amax/448,
        // code = E4M3(x * (448/amax)); all-zero rows get scale 1.
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(acc[c]));
        for (int o = G >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, o, G));
        float inv = 1.f, sc = 1.f;
        if (amax > 0.f) {
            inv = __fdiv_rn(448.f, amax);
            sc = __fdiv_rn(amax, 448.f);
        }
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(acc[4 * h], inv), __fmul_rn(acc[4 * h + 1], inv));
            uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(acc[4 * h + 2], inv), __fmul_rn(acc[4 * h + 3], inv));
            w[h] = lo | (hi << 16);
        }
        if (live) {
            *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) + r * d + 8 * g) = make_uint2(w[0], w[1]);
            if (g == 0) reinterpret_cast<float*>(out_scale)[r] = sc;
        }
    } else {
        // E2M1 codes with an E4M3 scale per 32 elements (4 threads):
        // sc = E4M3(amax/6) (at least the smallest positive E4M3), code = E2M1(x/sc).
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(acc[c]));
        const unsigned m4 = 0xFu << (lane & ~3u);
        amax = fmaxf(amax, __shfl_xor_sync(m4, amax, 1, 4));
        amax = fmaxf(amax, __shfl_xor_sync(m4, amax, 2, 4));
        uint32_t scc = f32x2_to_e4m3x2(__fdiv_rn(amax, 6.f), 0.f) & 0xFFu;
        if ((scc & 0x7Fu) == 0) scc = 0x01u;
        const float sc = e4m3x2_to_f32x2((uint16_t)scc).x;
        float y[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) y[c] = __fdiv_rn(acc[c], sc);
        const uint32_t packed = f32x8_to_e2m1x8(y);
        if (live) {
            reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(out) + r * (d / 2))[g] = packed;
            if ((g & 3) == 0) reinterpret_cast<uint8_t*>(out_scale)[r * (d / 32) + (g >> 2)] = (uint8_t)scc;
        }
    }
}

cudaError_t launch_compress(int B, int n, int m, int d, const float* logits, const void* x, bool x_bf16,
                            void* out, int out_kind, void* out_scale, cudaStream_t s)
{
    const int Nc = n / m;
    const long long threads = (long long)B * Nc * (d / 8);
    if (threads == 0) return cudaSuccess;
    const int bs = 256;
    const unsigned grid = (unsigned)((threads + bs - 1) / bs);
#define CSA_LAUNCH_COMPRESS(TIN, OK)                                                       \
    compress_kernel<TIN, OK><<<grid, bs, 0, s>>>(B, n, m, Nc, d, logits,                   \
                                                 reinterpret_cast<const TIN*>(x), out, out_scale)
    if (x_bf16) {
        switch (out_kind) {
            case 0: CSA_LAUNCH_COMPRESS(__nv_bfloat16, 0); break;
            case 1: CSA_LAUNCH_COMPRESS(__nv_bfloat16, 1); break;
            case 2: CSA_LAUNCH_COMPRESS(__nv_bfloat16, 2); break;
            default: CSA_LAUNCH_COMPRESS(__nv_bfloat16, 3); break;
        }
    } else {
        switch (out_kind) {
            case 0: CSA_LAUNCH_COMPRESS(float, 0); break;
            case 1: CSA_LAUNCH_COMPRESS(float, 1); break;
            case 2: CSA_LAUNCH_COMPRESS(float, 2); break;
            default: CSA_LAUNCH_COMPRESS(float, 3); break;
        }
    }
#undef CSA_LAUNCH_COMPRESS
    return cudaGetLastError();
}

}  // namespace csa
