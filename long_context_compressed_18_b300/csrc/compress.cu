// KV compression ("DeepSeek V4 技术解读" §2.1 KV Cache 压缩 and §2.2 HCA):
// every block of m raw tokens becomes one entry, the softmax-weighted sum of
// its tokens (one scalar logit per token).  Optional epilogues quantise the
// compressed entry to E4M3 (per-row fp32 scale) or E2M1 (E4M3 scale per 32
// elements) for the Lightning Indexer's FP8 / FP4 key cache.
//
// HBM-bound streaming reduction, two kernels.
//
// compress_tile_kernel (short blocks, m <= 32, every stream in one launch):
// persistent CTAs stream tiles of R consecutive entries through a shared-
// memory ring of about 64 KB with bulk async copies -- the tile's logits and, for each
// stream, its R*m contiguous input rows -- so the loads in flight per SM do not
// depend on registers.  A dedicated producer warp issues the copies; the block
// weights w_i = softmax(l)_i are computed once per entry (a group of lanes per
// entry, one lane per token) and shared by all streams, so the consumers'
// per-channel work is m FMAs.
//
// compress_kernel (long blocks, such as m' = 128, and shapes the bulk copies
// cannot take): one thread owns 8 consecutive channels of one output entry of
// one stream: it issues m 16-byte (bf16) or 2x16-byte (fp32) loads, coalesced
// across the G = d/8 threads of the row.
//
// In both, a thread accumulates its 8 channels in fp32 in token order (the
// long-block kernel divides by the softmax denominator at the end); row /
// block maxima for the quantisers are reduced across the row's thread group
// with shuffles.
#include "common.cuh"
#include "kernels.h"

namespace csa {

// Writes one thread's 8 compressed channels (acc, already divided by the
// softmax denominator) of output entry r: fp32 / bf16 as is, or quantised.  The
// G threads of the entry take part in the row / block maxima.  All 32 lanes of
// the warp call it together (dead lanes with live = false): the shuffles name
// the whole warp and stay inside their lane group through their width.
template <int OUT>
__device__ __forceinline__ void compress_store(const float (&acc)[8], int g, int G, long long r, int d, void* out,
                                               void* out_scale, bool live)
{
    if constexpr (OUT == 0 || OUT == 1) {
        using Tout = typename std::conditional<OUT == 0, float, __nv_bfloat16>::type;
        if (live) Vec8<Tout>::store(reinterpret_cast<Tout*>(out) + r * d + 8 * g, acc);
    } else if constexpr (OUT == 2) {
        // E4M3 codes with one fp32 scale per row: scale = amax/448,
        // code = E4M3(x * (448/amax)); all-zero rows get scale 1.
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(acc[c]));
        for (int o = G >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o, G));
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
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1, 4));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2, 4));
        uint32_t scc = f32x2_to_e4m3x2(__fdiv_rn(amax, 6.f), 0.f) & 0xFFu;
        if ((scc & 0x7Fu) == 0) scc = 0x01u;
        const float sc = e4m3x2_to_f32x2((uint16_t)scc).x;
        // x / sc correctly rounded without a division per element: the
        // correctly rounded reciprocal once, then q0 = |x| (1/sc) corrected
        // by one FMA residual step (Markstein's final step of FMA-based
        // division), the sign taken from x (so -0 and negatives that round to
        // zero keep their sign).  Compared with IEEE division over every fp32
        // significand of x and every positive E4M3 scale it never differs.
        const float rcp = __frcp_rn(sc);
        float y[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float ax = fabsf(acc[c]);
            const float q0 = __fmul_rn(ax, rcp);
            const float res = __fmaf_rn(-q0, sc, ax);
            y[c] = copysignf(__fmaf_rn(res, rcp, q0), acc[c]);
        }
        const uint32_t packed = f32x8_to_e2m1x8(y);
        if (live) {
            reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(out) + r * (d / 2))[g] = packed;
            if ((g & 3) == 0) reinterpret_cast<uint8_t*>(out_scale)[r * (d / 32) + (g >> 2)] = (uint8_t)scc;
        }
    }
}

// At most 64 registers a thread, so at least four CTAs (32 warps) share an SM.
// A CTA holds 256 / P threads per part: each of its P parts sums m / P of a
// block's tokens (in token order) for 256 / (P G) entries, and part 0 adds the
// parts' sums in part order.  P > 1 gives a short list of long blocks (few
// entries, m' = 128) enough threads to fill the GPU.
template <typename Tin, int OUT>
__global__ void __launch_bounds__(256, 4) compress_kernel(int B, int n, int m, int Nc, int d, int P,
                                                       const float* __restrict__ logits,
                                                       const Tin* __restrict__ x, void* out,
                                                       void* out_scale)
{
    grid_dep_entry();
    __shared__ float4 red[256][2];
    const int G = d >> 3;  // threads per output row (power of two, <= 32)
    const int TP = 256 / P, tid = threadIdx.x;
    const int part = tid / TP, t2 = tid - part * TP;
    const int g = t2 & (G - 1);
    const long long rows = (long long)B * Nc;
    const long long row = (long long)blockIdx.x * (TP / G) + t2 / G;
    const bool live = row < rows;
    const long long r = live ? row : rows - 1;  // dead lanes mirror the last row
    const long long b = r / Nc, j = r % Nc;

    // softmax statistics of the block's m logits, split across the row group
    const float* lg = logits + b * (long long)n + j * (long long)m;
    float mx = -INFINITY;
    for (int i = g; i < m; i += G) mx = fmaxf(mx, __ldg(lg + i));
    for (int o = G >> 1; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o, G));
    float den = 0.f;
    for (int i = g; i < m; i += G) den += expf(__ldg(lg + i) - mx);
    for (int o = G >> 1; o > 0; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o, G);

    // weighted sum over this part's tokens, in token order
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    const int mp = m / P, i0 = part * mp;
    const Tin* xp = x + (b * (long long)n + j * (long long)m) * d + 8 * g;
#pragma unroll 4
    for (int i = i0; i < i0 + mp; ++i) {
        float v[8];
        Vec8<Tin>::load(xp + (long long)i * d, v);
        const float e = expf(__ldg(lg + i) - mx);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = fmaf(e, v[c], acc[c]);
    }
    if (P > 1) {
        red[tid][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        red[tid][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        __syncthreads();
        if (part != 0) return;
        for (int q = 1; q < P; ++q) {
            const float4 u = red[q * TP + t2][0], w = red[q * TP + t2][1];
            acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
            acc[4] += w.x; acc[5] += w.y; acc[6] += w.z; acc[7] += w.w;
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = __fdiv_rn(acc[c], den);

    compress_store<OUT>(acc, g, G, r, d, out, out_scale, live);
}

cudaError_t launch_compress(int B, int n, int m, int d, const float* logits, const void* x, bool x_bf16,
                            void* out, int out_kind, void* out_scale, int num_sms, cudaStream_t s)
{
    const int Nc = n / m;
    const int G = d / 8;
    const long long threads = (long long)B * Nc * G;
    if (threads == 0) return cudaSuccess;
    // parts per block: while the GPU is not full, halve the tokens a thread
    // sums (at least 4 of them, the parts dividing m evenly)
    int P = 1;
    while (2 * P <= 8 && 2 * P * G <= 256 && m % (2 * P) == 0 && m / (2 * P) >= 4 && threads * P < (long long)num_sms * 512)
        P *= 2;
    const int bs = 256;
    const long long rows_per_cta = bs / P / G;
    const unsigned grid = (unsigned)((B * (long long)Nc + rows_per_cta - 1) / rows_per_cta);
#define CSA_LAUNCH_COMPRESS(TIN, OK)                                                       \
    (void)launch_pdl(compress_kernel<TIN, OK>, dim3(grid), dim3(bs), 0, s, B, n, m, Nc, d, P, logits,    \
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

// ---------------------------------------------------------------------------
// Per-channel compression weights (a variant reading of "weighted
// aggregation", "DeepSeek V4 技术解读" §2.1): every channel c has its own
// logit per token, logits [B, n, d], and
//     out[b, j, c] = sum_i softmax_i(logits[b, jm + i, c]) x[b, jm + i, c].
// One thread owns 8 consecutive channels of one entry: the block maxima, then
// the exponentials' sum and the weighted sum in token order, then the
// division -- fp32 throughout -- and the shared quantising epilogues.
// ---------------------------------------------------------------------------
template <typename Tin, int OUT>
__global__ void __launch_bounds__(256, 4) compress_channel_kernel(int B, int n, int m, int Nc, int d,
                                                               const float* __restrict__ logits,
                                                               const Tin* __restrict__ x, void* out,
                                                               void* out_scale)
{
    grid_dep_entry();
    const int G = d >> 3;   // threads per output row (power of two, <= 32)
    const long long rows = (long long)B * Nc;
    const long long row = (long long)blockIdx.x * (256 / G) + threadIdx.x / G;
    const int g = threadIdx.x & (G - 1);
    const bool live = row < rows;
    const long long r = live ? row : rows - 1;   // dead lanes mirror the last row
    const long long b = r / Nc, j = r % Nc;
    const long long base = (b * n + j * (long long)m) * d + 8 * g;
    float mx[8], den[8], acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        mx[c] = -INFINITY;
        den[c] = 0.f;
        acc[c] = 0.f;
    }
    for (int i = 0; i < m; ++i) {
        float l[8];
        Vec8<float>::load(logits + base + (long long)i * d, l);
#pragma unroll
        for (int c = 0; c < 8; ++c) mx[c] = fmaxf(mx[c], l[c]);
    }
    for (int i = 0; i < m; ++i) {
        float l[8], v[8];
        Vec8<float>::load(logits + base + (long long)i * d, l);
        Vec8<Tin>::load(x + base + (long long)i * d, v);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float e = expf(l[c] - mx[c]);
            den[c] += e;
            acc[c] = fmaf(e, v[c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = __fdiv_rn(acc[c], den[c]);
    compress_store<OUT>(acc, g, G, r, d, out, out_scale, live);
}

cudaError_t launch_compress_per_channel(int B, int n, int m, int d, const float* logits, const void* x, bool x_bf16,
                                        void* out, int out_kind, void* out_scale, cudaStream_t s)
{
    const int Nc = n / m;
    const long long rows = (long long)B * Nc;
    if (rows == 0) return cudaSuccess;
    const int rows_per_cta = 256 / (d / 8);
    const unsigned grid = (unsigned)((rows + rows_per_cta - 1) / rows_per_cta);
#define CSA_LAUNCH_CHANNEL(TIN, OK)                                                                  \
    (void)launch_pdl(compress_channel_kernel<TIN, OK>, dim3(grid), dim3(256), 0, s, B, n, m, Nc, d, logits,   \
                     reinterpret_cast<const TIN*>(x), out, out_scale)
    if (x_bf16) {
        switch (out_kind) {
            case 0: CSA_LAUNCH_CHANNEL(__nv_bfloat16, 0); break;
            case 1: CSA_LAUNCH_CHANNEL(__nv_bfloat16, 1); break;
            case 2: CSA_LAUNCH_CHANNEL(__nv_bfloat16, 2); break;
            default: CSA_LAUNCH_CHANNEL(__nv_bfloat16, 3); break;
        }
    } else {
        switch (out_kind) {
            case 0: CSA_LAUNCH_CHANNEL(float, 0); break;
            case 1: CSA_LAUNCH_CHANNEL(float, 1); break;
            case 2: CSA_LAUNCH_CHANNEL(float, 2); break;
            default: CSA_LAUNCH_CHANNEL(float, 3); break;
        }
    }
#undef CSA_LAUNCH_CHANNEL
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Short blocks: tiles of R entries x every stream, streamed by bulk copies.
// ---------------------------------------------------------------------------
namespace cmpt {
constexpr int CONSUMERS = 256;              // 8 warps: block weights, then the work items
constexpr int THREADS = CONSUMERS + 32;     // + one producer warp issuing the bulk copies
constexpr int MAX_STAGES = 8;
constexpr int RING_BUDGET = 65536;          // shared-memory ring per CTA
constexpr int MAX_M = 32;                   // one lane per token of a block
constexpr int MAX_R = 32;                   // entries per tile
constexpr int STAGE_BUDGET = 32768;         // two stages a ring
constexpr int ITEM_PASSES = 2;              // work items per consumer thread and tile, at most
constexpr int CTAS_PER_SM = 3;
}  // namespace cmpt

struct CompressTileStream {
    const void* x;
    void* out;
    void* out_scale;
    int d, es, in_bf16, kind;
    int lg_g;    // log2 of the threads per entry (d / 8)
    int soff;    // byte offset of this stream's rows inside a stage
    int item0;   // first work item of this stream (a multiple of 32)
};

struct CompressTileParams {
    const float* logits;
    int B, n, m, Nc, R, n_streams, tiles_per_b, n_tiles, stage_bytes, stages, items;
    CompressTileStream st[4];
};

__device__ __forceinline__ void lds8(const float* p, float (&v)[8])
{
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// acc[c] = sum_i w[i] * x[i][c] over the block's m tokens, in token order;
// xs points at this thread's 8 channels of the block's first token.
__device__ __forceinline__ void tile_accumulate_f32(const uint8_t* xs, int stride, const float* w, int m, float (&acc)[8])
{
#pragma unroll 4
    for (int i = 0; i < m; ++i) {
        float v[8];
        lds8(reinterpret_cast<const float*>(xs + (size_t)i * stride), v);
        const float e = w[i];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = fmaf(e, v[c], acc[c]);
    }
}

// bf16 inputs: channel pairs widened to fp32 pairs (low half: shift, high
// half: mask) and accumulated with paired FMAs.
__device__ __forceinline__ void tile_accumulate_bf16(const uint8_t* xs, int stride, const float* w, int m, float (&acc)[8])
{
    uint64_t a2[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) a2[c] = pack_f32x2(acc[2 * c], acc[2 * c + 1]);
#pragma unroll 4
    for (int i = 0; i < m; ++i) {
        const uint4 q = *reinterpret_cast<const uint4*>(xs + (size_t)i * stride);
        const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
        const float e = w[i];
        const uint64_t e2 = pack_f32x2(e, e);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            a2[c] = ffma2(e2, pack_u32x2(wq[c] << 16, wq[c] & 0xFFFF0000u), a2[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 f = unpack_f32x2(a2[c]);
        acc[2 * c] = f.x;
        acc[2 * c + 1] = f.y;
    }
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(cmpt::CONSUMERS) : "memory"); }

__global__ void __launch_bounds__(cmpt::THREADS, cmpt::CTAS_PER_SM)
compress_tile_kernel(const __grid_constant__ CompressTileParams p)
{
    grid_dep_entry();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ uint64_t full[cmpt::MAX_STAGES], empty[cmpt::MAX_STAGES];
    __shared__ float wts[2][cmpt::MAX_R * cmpt::MAX_M];   // by tile parity
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int R = p.R, m = p.m, S = p.stages;
    if (tid == 0) {
        for (int q = 0; q < S; ++q) {
            mbar_init(&full[q], 1);
            mbar_init(&empty[q], cmpt::CONSUMERS / 32);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // tile t -> batch b, first entry j0; entries [j0, j0 + re) of that batch
    auto tile_of = [&](int t, long long& row0, long long& tok0) {
        const int b = t / p.tiles_per_b, j0 = (t - b * p.tiles_per_b) * R;
        row0 = (long long)b * p.Nc + j0;
        tok0 = (long long)b * p.n + (long long)j0 * m;
        return min(R, p.Nc - j0);
    };

    if (warp == cmpt::CONSUMERS / 32) {
        // ---- producer: one lane streams the CTA's tiles into the ring ----
        if (lane != 0) return;
        int k = 0;
        for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++k) {
            const int slot = k % S;
            if (k >= S && !mbar_wait(&empty[slot], (uint32_t)(k / S - 1) & 1u, &abort_flag))
                break;
            long long row0, tok0;
            const int re = tile_of(t, row0, tok0);
            uint8_t* st = smem + (size_t)slot * p.stage_bytes;
            uint32_t bytes = (uint32_t)(re * m) * 4u;
            for (int s = 0; s < p.n_streams; ++s) bytes += (uint32_t)(re * m * p.st[s].d * p.st[s].es);
            mbar_arrive_expect_tx(&full[slot], bytes);
            bulk_load(st, p.logits + tok0, (uint32_t)(re * m) * 4u, &full[slot]);
            for (int s = 0; s < p.n_streams; ++s) {
                const CompressTileStream& sd = p.st[s];
                const size_t rb = (size_t)sd.d * sd.es;
                bulk_load(st + sd.soff, reinterpret_cast<const uint8_t*>(sd.x) + (size_t)tok0 * rb,
                          (uint32_t)((size_t)re * m * rb), &full[slot]);
            }
        }
        // copies still in flight into this CTA's shared memory land before
        // the CTA can exit (after an abort the consumers may have left)
        for (int q = k - S > 0 ? k - S : 0; q < k; ++q)
            mbar_wait(&full[q % S], (uint32_t)(q / S) & 1u);
        return;
    }

    // ---- consumers ----
    // weights: lanes in groups of gm (a power of two >= m), one entry a group
    const int gm = m <= 4 ? 4 : m <= 8 ? 8 : m <= 16 ? 16 : 32;
    const int per_warp = 32 / gm;
    const int gi = lane & (gm - 1);
    int k = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++k) {
        const int slot = k % S, par = k & 1;
        mbar_wait(&full[slot], (uint32_t)(k / S) & 1u, &abort_flag);
        const uint8_t* st = smem + (size_t)slot * p.stage_bytes;
        long long row0, tok0;
        const int re = tile_of(t, row0, tok0);

        // block weights w_i = exp(l_i - max) / sum_j exp(l_j - max)
        const float* lg = reinterpret_cast<const float*>(st);
        for (int r0 = warp * per_warp; r0 < re; r0 += (cmpt::CONSUMERS / 32) * per_warp) {
            const int r = r0 + lane / gm;
            const bool ok = r < re && gi < m;
            const float l = ok ? lg[r * m + gi] : -INFINITY;
            float mx = l;
            for (int o = gm >> 1; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o, gm));
            const float e = ok ? expf(l - mx) : 0.f;
            float sum = e;
            for (int o = gm >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o, gm);
            if (ok) wts[par][r * m + gi] = __fdiv_rn(e, sum);
        }
        consumer_sync();
        if (abort_flag) break;

        // work items: (stream, entry r, 8-channel group g); a stream's items
        // start at a multiple of 32, so a warp never mixes streams; lanes past
        // the tile's entries mirror its last entry and store nothing
        for (int item = tid; item < p.items; item += cmpt::CONSUMERS) {
            int s = 0;
            while (s + 1 < p.n_streams && item >= p.st[s + 1].item0) ++s;
            const CompressTileStream& sd = p.st[s];
            const int G = sd.d >> 3;
            const int local = item - sd.item0;
            const int rr = local >> sd.lg_g, g = local & (G - 1);
            const bool live = rr < re;
            const int r = live ? rr : re - 1;
            const int stride = sd.d * sd.es;
            const uint8_t* xs = st + sd.soff + (size_t)r * m * stride + (size_t)8 * g * sd.es;
            float acc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = 0.f;
            if (sd.in_bf16) tile_accumulate_bf16(xs, stride, wts[par] + r * m, m, acc);
            else tile_accumulate_f32(xs, stride, wts[par] + r * m, m, acc);
            const long long row = row0 + r;
            switch (sd.kind) {
                case 0: compress_store<0>(acc, g, G, row, sd.d, sd.out, sd.out_scale, live); break;
                case 1: compress_store<1>(acc, g, G, row, sd.d, sd.out, sd.out_scale, live); break;
                case 2: compress_store<2>(acc, g, G, row, sd.d, sd.out, sd.out_scale, live); break;
                default: compress_store<3>(acc, g, G, row, sd.d, sd.out, sd.out_scale, live); break;
            }
        }
        // this warp is done with the stage; the weights buffer of this
        // tile's parity is rewritten only after the next tile's barrier
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

bool compress_tiles_supported(int n, int m, int n_streams, const int* dim, const bool* x_bf16)
{
    if (m < 4 || m > cmpt::MAX_M || (m & 3) || (n & 3) || n_streams < 1 || n_streams > 4) return false;
    int row = align_up(m * 4, 128), items = 0;
    for (int s = 0; s < n_streams; ++s) {
        row += align_up(m * dim[s] * (x_bf16[s] ? 2 : 4), 128);
        items += align_up(dim[s] / 8, 32);
    }
    return row <= cmpt::STAGE_BUDGET && items <= cmpt::CONSUMERS;
}

cudaError_t launch_compress_tiles(int B, int n, int m, int n_streams, const float* logits, const void* const* x,
                                  const bool* x_bf16, const int* dim, void* const* out, const int* out_kind,
                                  void* const* out_scale, int num_sms, cudaStream_t s)
{
    const int Nc = n / m;
    if ((long long)B * Nc == 0) return cudaSuccess;
    auto stage_of = [&](int R) {
        int b = align_up(R * m * 4, 128);
        for (int q = 0; q < n_streams; ++q) b += align_up(R * m * dim[q] * (x_bf16[q] ? 2 : 4), 128);
        return b;
    };
    // the largest tile whose stage fits the budget and whose work items fit
    // two passes of the consumer threads: large tiles spread the per-tile
    // steps (barrier waits, the block weights, the bulk-copy issue) over more
    // entries (three streams at m = 4: R = 10, 480 items; 56 -> 70 % of HBM
    // against R = 4 in one pass)
    auto items_of = [&](int R) {
        int it = 0;
        for (int q = 0; q < n_streams; ++q) it += align_up(R * (dim[q] / 8), 32);
        return it;
    };
    int R = cmpt::MAX_R;
    while (R > 1 && (stage_of(R) > cmpt::STAGE_BUDGET || items_of(R) > cmpt::ITEM_PASSES * cmpt::CONSUMERS)) --R;
    const long long slots = (long long)num_sms * cmpt::CTAS_PER_SM;
    CompressTileParams p{};
    p.logits = logits;
    p.B = B; p.n = n; p.m = m; p.Nc = Nc; p.R = R; p.n_streams = n_streams;
    p.tiles_per_b = (Nc + R - 1) / R;
    const long long n_tiles = (long long)B * p.tiles_per_b;
    if (n_tiles > INT32_MAX) return cudaErrorInvalidValue;
    p.n_tiles = (int)n_tiles;
    int off = align_up(R * m * 4, 128), item = 0;
    for (int q = 0; q < n_streams; ++q) {
        CompressTileStream& sd = p.st[q];
        sd.x = x[q]; sd.out = out[q]; sd.out_scale = out_scale ? out_scale[q] : nullptr;
        sd.d = dim[q]; sd.es = x_bf16[q] ? 2 : 4; sd.in_bf16 = x_bf16[q] ? 1 : 0; sd.kind = out_kind[q];
        sd.lg_g = 0;
        while ((8 << sd.lg_g) < dim[q]) ++sd.lg_g;
        sd.soff = off; sd.item0 = item;
        off += align_up(R * m * dim[q] * sd.es, 128);
        item += align_up(R * (dim[q] / 8), 32);
    }
    p.stage_bytes = off;
    p.stages = cmpt::RING_BUDGET / off < 2 ? 2 : cmpt::RING_BUDGET / off > cmpt::MAX_STAGES ? cmpt::MAX_STAGES
                                                                                          : cmpt::RING_BUDGET / off;
    p.items = item;
    const int smem = p.stages * p.stage_bytes;
    cudaError_t e = cudaFuncSetAttribute(compress_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(n_tiles < slots ? n_tiles : slots);
    (void)launch_pdl(compress_tile_kernel, dim3(grid), dim3(cmpt::THREADS), smem, s, p);
    return cudaGetLastError();
}

}  // namespace csa
