// Streaming decode state: the KV-cache compression of "DeepSeek V4 技术解读"
// §2.1 (KV Cache 压缩: every m tokens' KV entries merged into one entry by
// weighted aggregation) applied one generated token at a time.
//
// Each sequence keeps its last, still open block of raw tokens in a staging
// buffer.  Appending a token writes it into its slot of that buffer and
// advances the sequence's token count (a device array, so a decode loop needs
// no host round trip); when the token closes the block (count % m == 0) the
// block is compressed into the next entry of the sequence's caches -- K_c,
// V_c and the indexer keys, quantised to E4M3 or E2M1 as the caches are kept
// -- with the same arithmetic as csa_compress: weights w_i = softmax of the
// block's logits, fp32 sums in token order, then the quantising epilogue.
#include "common.cuh"
#include "kernels.h"

namespace csa {

constexpr int APPEND_THREADS = 128;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// One CTA per sequence.
template <typename TIN>
__global__ void __launch_bounds__(APPEND_THREADS) decode_append_kernel(DecodeAppendArgs a)
{
    grid_dep_entry();
    __shared__ float w[DECODE_MAX_M];
    __shared__ float row[256];
    __shared__ float red[APPEND_THREADS / 32];
    __shared__ long long t_s;
    const int b = blockIdx.x, tid = threadIdx.x;
    if (tid == 0) t_s = a.lens[b];
    __syncthreads();
    const long long t = t_s;                       // tokens before this one
    if (t < 0) {                                   // a corrupt count: touch nothing
        if (tid == 0) flag_status(STATUS_BOUNDS);
        return;
    }
    const int slot = (int)(t % a.m);
    const TIN* kn = reinterpret_cast<const TIN*>(a.k_new) + (long long)b * a.d;
    const TIN* vn = reinterpret_cast<const TIN*>(a.v_new) + (long long)b * a.d;
    const TIN* in = reinterpret_cast<const TIN*>(a.ik_new) + (long long)b * a.d_I;
    TIN* sk = reinterpret_cast<TIN*>(a.st_k) + ((long long)b * a.m + slot) * a.d;
    TIN* sv = reinterpret_cast<TIN*>(a.st_v) + ((long long)b * a.m + slot) * a.d;
    TIN* si = reinterpret_cast<TIN*>(a.st_ik) + ((long long)b * a.m + slot) * a.d_I;
    for (int c = tid; c < a.d; c += APPEND_THREADS) {
        sk[c] = kn[c];
        sv[c] = vn[c];
    }
    for (int c = tid; c < a.d_I; c += APPEND_THREADS) si[c] = in[c];
    if (tid == 0) a.st_logit[(long long)b * a.m + slot] = a.logit_new[b];
    __syncthreads();                               // the staged block is complete and visible
    if ((t + 1) % a.m == 0) {
        const long long j = (t + 1) / a.m - 1;     // the entry this block becomes
        if (j >= a.N_cap) {
            if (tid == 0) flag_status(STATUS_BOUNDS);
        } else {
            // block weights: softmax of the m staged logits
            const float* lg = a.st_logit + (long long)b * a.m;
            float mx = -INFINITY;
            for (int i = 0; i < a.m; ++i) mx = fmaxf(mx, lg[i]);
            float den = 0.f;
            for (int i = 0; i < a.m; ++i) den += expf(lg[i] - mx);
            for (int i = tid; i < a.m; i += APPEND_THREADS) w[i] = __fdiv_rn(expf(lg[i] - mx), den);
            __syncthreads();
            auto compress_row = [&](const TIN* stage, int d, int c) {
                float acc = 0.f;
                for (int i = 0; i < a.m; ++i) acc = fmaf(w[i], to_f32(stage[(long long)i * d + c]), acc);
                return acc;
            };
            const TIN* bk = reinterpret_cast<const TIN*>(a.st_k) + (long long)b * a.m * a.d;
            const TIN* bv = reinterpret_cast<const TIN*>(a.st_v) + (long long)b * a.m * a.d;
            const TIN* bi = reinterpret_cast<const TIN*>(a.st_ik) + (long long)b * a.m * a.d_I;
            const long long e = (long long)b * a.N_cap + j;
            for (int c = tid; c < a.d; c += APPEND_THREADS) {
                const float kc = compress_row(bk, a.d, c), vc = compress_row(bv, a.d, c);
                if (a.kv_kind == 0) {
                    reinterpret_cast<float*>(a.k_c)[e * a.d + c] = kc;
                    reinterpret_cast<float*>(a.v_c)[e * a.d + c] = vc;
                } else {
                    reinterpret_cast<__nv_bfloat16*>(a.k_c)[e * a.d + c] = __float2bfloat16_rn(kc);
                    reinterpret_cast<__nv_bfloat16*>(a.v_c)[e * a.d + c] = __float2bfloat16_rn(vc);
                }
            }
            for (int c = tid; c < a.d_I; c += APPEND_THREADS) row[c] = compress_row(bi, a.d_I, c);
            __syncthreads();
            // the indexer-key epilogue (the quantisers of csa_compress)
            if (a.ik_kind == 0 || a.ik_kind == 1) {
                for (int c = tid; c < a.d_I; c += APPEND_THREADS) {
                    if (a.ik_kind == 0) reinterpret_cast<float*>(a.ik_c)[e * a.d_I + c] = row[c];
                    else reinterpret_cast<__nv_bfloat16*>(a.ik_c)[e * a.d_I + c] = __float2bfloat16_rn(row[c]);
                }
            } else if (a.ik_kind == 2) {
                // E4M3 codes, one fp32 scale: scale = amax/448, code = E4M3(x * (448/amax))
                float amax = 0.f;
                for (int c = tid; c < a.d_I; c += APPEND_THREADS) amax = fmaxf(amax, fabsf(row[c]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                if ((tid & 31) == 0) red[tid >> 5] = amax;
                __syncthreads();
                amax = 0.f;
                for (int q = 0; q < APPEND_THREADS / 32; ++q) amax = fmaxf(amax, red[q]);
                float inv = 1.f, sc = 1.f;
                if (amax > 0.f) {
                    inv = __fdiv_rn(448.f, amax);
                    sc = __fdiv_rn(amax, 448.f);
                }
                uint8_t* codes = reinterpret_cast<uint8_t*>(a.ik_c) + e * a.d_I;
                for (int c = 2 * tid; c < a.d_I; c += 2 * APPEND_THREADS) {
                    const uint16_t two = f32x2_to_e4m3x2(__fmul_rn(row[c], inv), __fmul_rn(row[c + 1], inv));
                    codes[c] = (uint8_t)(two & 0xFFu);
                    codes[c + 1] = (uint8_t)(two >> 8);
                }
                if (tid == 0) reinterpret_cast<float*>(a.ik_scale)[e] = sc;
            } else {
                // E2M1 codes with an E4M3 scale per 32 elements: sc = E4M3(amax/6)
                // (at least the smallest positive E4M3), code = E2M1(x / sc)
                const int nb = a.d_I / 32;
                for (int blk = tid; blk < nb; blk += APPEND_THREADS) {
                    float amax = 0.f;
                    for (int c = 0; c < 32; ++c) amax = fmaxf(amax, fabsf(row[blk * 32 + c]));
                    uint32_t scc = f32x2_to_e4m3x2(__fdiv_rn(amax, 6.f), 0.f) & 0xFFu;
                    if ((scc & 0x7Fu) == 0) scc = 0x01u;
                    const float sc = e4m3x2_to_f32x2((uint16_t)scc).x;
                    uint32_t* packed = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(a.ik_c) + e * (a.d_I / 2) +
                                                                   blk * 16);
                    for (int q = 0; q < 4; ++q) {
                        float y[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) y[c] = __fdiv_rn(row[blk * 32 + 8 * q + c], sc);
                        packed[q] = f32x8_to_e2m1x8(y);
                    }
                    reinterpret_cast<uint8_t*>(a.ik_scale)[e * nb + blk] = (uint8_t)scc;
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) a.lens[b] = t + 1;
}

cudaError_t launch_decode_append(const DecodeAppendArgs& a, bool x_bf16, cudaStream_t s)
{
    if (a.B == 0) return cudaSuccess;
    if (x_bf16) (void)launch_pdl(decode_append_kernel<__nv_bfloat16>, dim3(a.B), dim3(APPEND_THREADS), 0, s, a);
    else (void)launch_pdl(decode_append_kernel<float>, dim3(a.B), dim3(APPEND_THREADS), 0, s, a);
    return cudaGetLastError();
}

}  // namespace csa
