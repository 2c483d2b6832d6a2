// Top-k selection ("DeepSeek V4 技术解读" §2.1: the Lightning Indexer keeps the
// k highest-scoring compressed entries per query).
//
// Exact radix select on order-preserving 32-bit keys of the fp32 scores
// (-0 folded onto +0).  A CTA stages its elements' keys in shared memory,
// finds the k-th largest key T with three histogram levels (11, 11 and 10
// bits; see radix_threshold), then writes
// the selected indices in ascending order with a warp-ballot compaction:
// every key > T, plus the first (k - #{key > T}) elements equal to T in index
// order -- i.e. ranking by (score desc, index asc).  No floating-point
// atomics; the result does not depend on thread scheduling.
//
// Rows longer than one CTA's capacity are split: phase A selects the top-k of
// each chunk (candidates keep ascending index order), phase B selects from
// the concatenated candidates.  The global top-k is contained in the union of
// the chunk top-k sets, so the result is identical to a single pass.
#include "common.cuh"
#include "kernels.h"

namespace csa {

constexpr int TOPK_THREADS = 512;
constexpr int TOPK_WARPS = TOPK_THREADS / 32;

__device__ __forceinline__ uint32_t score_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;                               // -0 -> +0
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;           // NaN ranks last
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Radix levels over the 32-bit key: bits 31..21 (2048 bins), 20..10 (2048),
// 9..0 (1024).  The first level's histogram is built while the scores are
// loaded; the second while the elements of the selected first-level bin are
// compacted into a candidate list, so only that (short) list is scanned for
// the third level.  Rows whose selected bin overflows the list (heavy ties)
// scan the full key array instead.
constexpr int CAND_CAP = 2048;

struct TopkShared {
    uint32_t hist[2048];
    uint32_t cand[CAND_CAP];
    uint32_t scan[TOPK_WARPS];
    uint32_t warp_take[TOPK_WARPS];
    uint32_t warp_eq[TOPK_WARPS];
    uint32_t n_cand, bin, above;
};

__device__ __forceinline__ void clear_hist(TopkShared& sh, int nb)
{
    for (int i = threadIdx.x; i < nb; i += TOPK_THREADS) sh.hist[i] = 0;
}

// Scanning the NB-bin histogram from the top bin down, finds the bin in which
// the running count reaches rem (1 <= rem <= total): sh.bin = that bin,
// sh.above = the count of all higher bins (< rem).
template <int NB>
__device__ void find_bin(TopkShared& sh, uint32_t rem)
{
    constexpr int BPT = NB / TOPK_THREADS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t c[BPT], tot = 0;
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        c[q] = sh.hist[NB - 1 - tid * BPT - q];
        tot += c[q];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) sh.scan[warp] = incl;
    __syncthreads();
    uint32_t before = incl - tot;
    for (int w = 0; w < warp; ++w) before += sh.scan[w];
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        if (before < rem && before + c[q] >= rem) {
            sh.bin = (uint32_t)(NB - 1 - tid * BPT - q);
            sh.above = before;
        }
        before += c[q];
    }
    __syncthreads();
}

// The k-th largest key T among keys[0..len) and how many elements equal to T
// are selected (take_eq), for 1 <= kk <= len.  Requires sh.hist to hold the
// first-level histogram (key >> 21) of keys[0..len).
__device__ void radix_threshold(const uint32_t* keys, int len, int kk, TopkShared& sh, uint32_t& T_out,
                                int& take_eq_out)
{
    const int tid = threadIdx.x, lane = tid & 31;
    find_bin<2048>(sh, (uint32_t)kk);
    const uint32_t b1 = sh.bin;
    uint32_t rem = (uint32_t)kk - sh.above;
    clear_hist(sh, 2048);
    if (tid == 0) sh.n_cand = 0;
    __syncthreads();
    // candidates of bin b1 (their order is irrelevant: only T and take_eq are
    // derived from them) and the second-level histogram
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < len; base += TOPK_THREADS) {
        const int e = base + tid;
        const uint32_t key = e < len ? keys[e] : 0u;
        const bool m = e < len && (key >> 21) == b1;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
        uint32_t pos0 = 0;
        if (lane == 0 && bal) pos0 = atomicAdd(&sh.n_cand, (uint32_t)__popc(bal));
        pos0 = __shfl_sync(0xFFFFFFFFu, pos0, 0);
        if (m) {
            const uint32_t pos = pos0 + __popc(bal & lt);
            if (pos < CAND_CAP) sh.cand[pos] = key;
            atomicAdd(&sh.hist[(key >> 10) & 0x7FFu], 1u);
        }
    }
    __syncthreads();
    find_bin<2048>(sh, rem);
    const uint32_t pre = (b1 << 11) | sh.bin;     // required value of key >> 10
    rem -= sh.above;
    const int nc = (int)sh.n_cand;
    clear_hist(sh, 1024);
    __syncthreads();
    const uint32_t* src = nc <= CAND_CAP ? sh.cand : keys;
    const int n = nc <= CAND_CAP ? nc : len;
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const uint32_t key = src[e];
        if ((key >> 10) == pre) atomicAdd(&sh.hist[key & 0x3FFu], 1u);
    }
    __syncthreads();
    find_bin<1024>(sh, rem);
    T_out = (pre << 10) | sh.bin;
    take_eq_out = (int)(rem - sh.above);
}

// Loads len fp32 scores into shared memory as keys and accumulates the
// first-level histogram.  Each thread keeps eight loads in flight.
__device__ void load_score_keys(const float* __restrict__ src, int len, uint32_t* keys, TopkShared& sh)
{
    const int tid = threadIdx.x;
    constexpr int U = 8;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const int n4 = len >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(src);
        for (int base = 0; base < n4; base += TOPK_THREADS * U) {
            float4 f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = base + u * TOPK_THREADS + tid;
                f[u] = v < n4 ? __ldg(s4 + v) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = base + u * TOPK_THREADS + tid;
                if (v < n4) {
                    const uint4 kq = make_uint4(score_key(f[u].x), score_key(f[u].y), score_key(f[u].z),
                                                score_key(f[u].w));
                    reinterpret_cast<uint4*>(keys)[v] = kq;
                    atomicAdd(&sh.hist[kq.x >> 21], 1u);
                    atomicAdd(&sh.hist[kq.y >> 21], 1u);
                    atomicAdd(&sh.hist[kq.z >> 21], 1u);
                    atomicAdd(&sh.hist[kq.w >> 21], 1u);
                }
            }
        }
        for (int e = 4 * n4 + tid; e < len; e += TOPK_THREADS) {
            const uint32_t key = score_key(__ldg(src + e));
            keys[e] = key;
            atomicAdd(&sh.hist[key >> 21], 1u);
        }
    } else {
        for (int base = 0; base < len; base += TOPK_THREADS * U) {
            float f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                f[u] = e < len ? __ldg(src + e) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                if (e < len) {
                    const uint32_t key = score_key(f[u]);
                    keys[e] = key;
                    atomicAdd(&sh.hist[key >> 21], 1u);
                }
            }
        }
    }
}

// Ordered compaction: selected(e) = key > T || (key == T && eq-rank(e) < take_eq).
// emit(pos, e) is called once per selected element with its output slot.
template <typename Emit>
__device__ void ordered_compact(const uint32_t* keys, int len, uint32_t T, int take_eq,
                                TopkShared& sh, Emit emit)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (((len + TOPK_WARPS - 1) / TOPK_WARPS) + 31) & ~31;
    const int lo = min(len, warp * per), hi = min(len, lo + per);
    uint32_t n_take = 0, n_eq = 0;
    for (int e0 = lo; e0 < hi; e0 += 32) {
        const int e = e0 + lane;
        const uint32_t key = e < hi ? keys[e] : 0u;
        n_take += __popc(__ballot_sync(0xFFFFFFFFu, e < hi && key > T));
        n_eq += __popc(__ballot_sync(0xFFFFFFFFu, e < hi && key == T));
    }
    if (lane == 0) { sh.warp_take[warp] = n_take; sh.warp_eq[warp] = n_eq; }
    __syncthreads();
    uint32_t take_base = 0, eq_base = 0, eq_total_before = 0;
    for (int w = 0; w < warp; ++w) eq_total_before += sh.warp_eq[w];
    // equal elements taken by earlier warps
    {
        uint32_t eq_taken_before = min(eq_total_before, (uint32_t)take_eq);
        for (int w = 0; w < warp; ++w) take_base += sh.warp_take[w];
        take_base += eq_taken_before;
        eq_base = eq_total_before;
    }
    const unsigned lt = (1u << lane) - 1u;
    for (int e0 = lo; e0 < hi; e0 += 32) {
        const int e = e0 + lane;
        const uint32_t key = e < hi ? keys[e] : 0u;
        const unsigned bgt = __ballot_sync(0xFFFFFFFFu, e < hi && key > T);
        const unsigned beq = __ballot_sync(0xFFFFFFFFu, e < hi && key == T);
        const uint32_t my_eq_rank = eq_base + __popc(beq & lt);
        const bool eq_sel = (beq >> lane & 1u) && my_eq_rank < (uint32_t)take_eq;
        const unsigned bsel = bgt | __ballot_sync(0xFFFFFFFFu, eq_sel);
        if (bsel >> lane & 1u) emit((int)(take_base + __popc(bsel & lt)), e);
        take_base += __popc(bsel);
        eq_base += __popc(beq);
    }
}

// MODE 0: fp32 score rows.  Each CTA handles chunk c of row r.  With
//         n_chunks == 1 it writes the final indices (-1 padded); otherwise it
//         writes min(k, chunk_len) candidates (key, index) for phase B.
// MODE 1: phase B over the candidates of a row.  Every chunk but the last
//         non-empty one contributes exactly k candidates, so a row's
//         candidates are one contiguous run of its [n_chunks, k] buffer.
template <int MODE>
__global__ void __launch_bounds__(TOPK_THREADS) topk_kernel(
    const float* __restrict__ scores, long long ld, int n_q_rows, long long q_pos0, int m, int Nc,
    int k, int chunk, int n_chunks, uint32_t* cand_key, int32_t* cand_idx, int32_t* __restrict__ out,
    long long out_b_stride)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ TopkShared sh;
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);
    // phase A / single pass: one CTA per (row, chunk); phase B: one CTA per row
    const int r = (MODE == 0) ? (int)(blockIdx.x / n_chunks) : (int)blockIdx.x;
    const int c = (MODE == 0) ? (int)(blockIdx.x % n_chunks) : 0;
    const int i = r % n_q_rows;   // query index within the chunk of rows
    const long long out_row = (long long)(r / n_q_rows) * out_b_stride + i;
    long long nvl = (q_pos0 + i + 1) / m;
    const int L = (int)(nvl < Nc ? nvl : Nc);
    const int tid = threadIdx.x;
    clear_hist(sh, 2048);
    __syncthreads();

    if constexpr (MODE == 0) {
        const int c0 = c * chunk;
        const int len = max(0, min(chunk, L - c0));
        const float* row = scores + (long long)r * ld + c0;
        const int kk = min(k, len);
        if (n_chunks == 1) {
            int32_t* o = out + out_row * k;
            for (int p = kk + tid; p < k; p += TOPK_THREADS) o[p] = -1;
            if (kk == 0) return;
            if (len <= k) {
                for (int e = tid; e < len; e += TOPK_THREADS) o[e] = e;
                return;
            }
            load_score_keys(row, len, keys, sh);
            __syncthreads();
            uint32_t T; int teq;
            radix_threshold(keys, len, kk, sh, T, teq);
            ordered_compact(keys, len, T, teq, sh, [&](int pos, int e) { if (pos < kk) o[pos] = e; });
        } else {
            uint32_t* ck = cand_key + ((long long)r * n_chunks + c) * k;
            int32_t* ci = cand_idx + ((long long)r * n_chunks + c) * k;
            if (kk == 0) return;
            if (len <= k) {
                for (int e = tid; e < len; e += TOPK_THREADS) { ck[e] = score_key(row[e]); ci[e] = c0 + e; }
                return;
            }
            load_score_keys(row, len, keys, sh);
            __syncthreads();
            uint32_t T; int teq;
            radix_threshold(keys, len, kk, sh, T, teq);
            ordered_compact(keys, len, T, teq, sh, [&](int pos, int e) {
                if (pos < kk) { ck[pos] = keys[e]; ci[pos] = c0 + e; }
            });
        }
    } else {
        int32_t* idxs = reinterpret_cast<int32_t*>(keys + (long long)n_chunks * k);
        int total = 0;
        for (int cc = 0; cc < n_chunks; ++cc) total += min(k, max(0, min(chunk, L - cc * chunk)));
        const uint32_t* ck = cand_key + (long long)r * n_chunks * k;
        const int32_t* ci = cand_idx + (long long)r * n_chunks * k;
        constexpr int U = 8;
        for (int base = 0; base < total; base += TOPK_THREADS * U) {
            uint32_t kv[U];
            int32_t iv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                kv[u] = e < total ? __ldg(ck + e) : 0u;
                iv[u] = e < total ? __ldg(ci + e) : 0;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                if (e < total) {
                    keys[e] = kv[u];
                    idxs[e] = iv[u];
                    atomicAdd(&sh.hist[kv[u] >> 21], 1u);
                }
            }
        }
        __syncthreads();
        int32_t* o = out + out_row * k;
        const int kk = min(k, total);
        for (int p = kk + tid; p < k; p += TOPK_THREADS) o[p] = -1;
        if (kk == 0) return;
        if (total <= k) {
            for (int e = tid; e < total; e += TOPK_THREADS) o[e] = idxs[e];
            return;
        }
        uint32_t T; int teq;
        radix_threshold(keys, total, kk, sh, T, teq);
        ordered_compact(keys, total, T, teq, sh, [&](int pos, int e) { if (pos < kk) o[pos] = idxs[e]; });
    }
}

// Chunking plan shared by the launcher and the workspace query.
TopkPlan topk_plan(int N_c, int k)
{
    TopkPlan p;
    if (N_c <= TOPK_MAX_SINGLE) {
        p.chunk = N_c > 0 ? N_c : 1;
        p.n_chunks = 1;
    } else {
        int chunk = 16384;
        while ((N_c + chunk - 1) / chunk * k > TOPK_MAX_MERGE && chunk < TOPK_MAX_SINGLE) chunk *= 2;
        p.chunk = chunk;
        p.n_chunks = (N_c + chunk - 1) / chunk;
    }
    return p;
}

size_t topk_workspace_bytes(int rows, int N_c, int k)
{
    TopkPlan p = topk_plan(N_c, k);
    if (p.n_chunks == 1) return 0;
    return (size_t)rows * p.n_chunks * k * (sizeof(uint32_t) + sizeof(int32_t));
}

cudaError_t launch_topk(const float* scores, long long ld, int B, int n_q_rows, long long q_pos0,
                        int m, int N_c, int k, int32_t* out, long long out_b_stride, void* ws,
                        cudaStream_t s)
{
    const int rows = B * n_q_rows;
    if (rows == 0) return cudaSuccess;
    TopkPlan p = topk_plan(N_c, k);
    if (p.n_chunks == 1) {
        size_t smem = (size_t)p.chunk * sizeof(uint32_t);
        auto kern = topk_kernel<0>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<rows, TOPK_THREADS, smem, s>>>(scores, ld, n_q_rows, q_pos0, m, N_c, k, p.chunk, 1,
                                              nullptr, nullptr, out, out_b_stride);
        return cudaGetLastError();
    }
    uint32_t* ck = reinterpret_cast<uint32_t*>(ws);
    int32_t* ci = reinterpret_cast<int32_t*>(ck + (size_t)rows * p.n_chunks * k);
    {
        size_t smem = (size_t)p.chunk * sizeof(uint32_t);
        auto kern = topk_kernel<0>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<rows * p.n_chunks, TOPK_THREADS, smem, s>>>(scores, ld, n_q_rows, q_pos0, m, N_c, k,
                                                           p.chunk, p.n_chunks, ck, ci, out, out_b_stride);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    {
        size_t smem = (size_t)p.n_chunks * k * (sizeof(uint32_t) + sizeof(int32_t));
        auto kern = topk_kernel<1>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<rows, TOPK_THREADS, smem, s>>>(scores, ld, n_q_rows, q_pos0, m, N_c, k, p.chunk,
                                              p.n_chunks, ck, ci, out, out_b_stride);
    }
    return cudaGetLastError();
}

}  // namespace csa
