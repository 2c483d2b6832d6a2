// Top-k selection ("DeepSeek V4 技术解读" §2.1: the Lightning Indexer keeps the
// k highest-scoring compressed entries per query).
//
// Exact radix select on order-preserving 32-bit keys of the fp32 scores
// (-0 folded onto +0).  A CTA stages its elements' keys in shared memory,
// finds the k-th largest key T with four 8-bit histogram passes, then writes
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

struct TopkShared {
    uint32_t hist[256];
    uint32_t warp_take[TOPK_WARPS];
    uint32_t warp_eq[TOPK_WARPS];
    uint32_t digit, above;
};

// Finds T (the k-th largest key among keys[0..len)) and how many elements
// equal to T are selected.  Requires 1 <= kk <= len.
__device__ void radix_threshold(const uint32_t* keys, int len, int kk, TopkShared& sh,
                                uint32_t& T_out, int& take_eq_out)
{
    uint32_t prefix = 0;
    int remaining = kk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t himask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        for (int i = tid; i < 256; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < len; base += blockDim.x) {
            const int e = base + tid;
            const bool in = e < len && ((keys[e] & himask) == prefix);
            const uint32_t dig = in ? ((keys[e] >> shift) & 255u) : 256u;
            // aggregate equal digits within the warp before the shared atomic
            const unsigned peers = __match_any_sync(0xFFFFFFFFu, dig);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[dig], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (descending); suffix counts from the top
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) { c[q] = sh.hist[255 - 8 * lane - q]; tot += c[q]; }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            uint32_t above = incl - tot;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (above < (uint32_t)remaining && above + c[q] >= (uint32_t)remaining) {
                    sh.digit = 255u - 8u * lane - q;
                    sh.above = above;
                }
                above += c[q];
            }
        }
        __syncthreads();
        prefix |= sh.digit << shift;
        remaining -= (int)sh.above;
        __syncthreads();
    }
    T_out = prefix;
    take_eq_out = remaining;
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
// MODE 1: phase B over the candidates of a row.
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

    if constexpr (MODE == 0) {
        const int c0 = c * chunk;
        const int len = max(0, min(chunk, L - c0));
        const float* row = scores + (long long)r * ld + c0;
        for (int e = tid; e < len; e += blockDim.x) keys[e] = score_key(row[e]);
        __syncthreads();
        const int kk = min(k, len);
        if (n_chunks == 1) {
            int32_t* o = out + out_row * k;
            for (int p = kk + tid; p < k; p += blockDim.x) o[p] = -1;
            if (kk == 0) return;
            if (len <= k) {
                for (int e = tid; e < len; e += blockDim.x) o[e] = e;
                return;
            }
            uint32_t T; int teq;
            radix_threshold(keys, len, kk, sh, T, teq);
            ordered_compact(keys, len, T, teq, sh, [&](int pos, int e) { o[pos] = e; });
        } else {
            uint32_t* ck = cand_key + ((long long)r * n_chunks + c) * k;
            int32_t* ci = cand_idx + ((long long)r * n_chunks + c) * k;
            if (kk == 0) return;
            if (len <= k) {
                for (int e = tid; e < len; e += blockDim.x) { ck[e] = keys[e]; ci[e] = c0 + e; }
                return;
            }
            uint32_t T; int teq;
            radix_threshold(keys, len, kk, sh, T, teq);
            ordered_compact(keys, len, T, teq, sh, [&](int pos, int e) { ck[pos] = keys[e]; ci[pos] = c0 + e; });
        }
    } else {
        // gather this row's candidates in chunk order (ascending entry index)
        int32_t* idxs = reinterpret_cast<int32_t*>(keys + (long long)n_chunks * k);
        int total = 0;
        for (int cc = 0; cc < n_chunks; ++cc) {
            const int len_c = max(0, min(chunk, L - cc * chunk));
            const int cnt = min(k, len_c);
            const uint32_t* ck = cand_key + ((long long)r * n_chunks + cc) * k;
            const int32_t* ci = cand_idx + ((long long)r * n_chunks + cc) * k;
            for (int e = tid; e < cnt; e += blockDim.x) { keys[total + e] = ck[e]; idxs[total + e] = ci[e]; }
            total += cnt;
        }
        __syncthreads();
        int32_t* o = out + out_row * k;
        const int kk = min(k, total);
        for (int p = kk + tid; p < k; p += blockDim.x) o[p] = -1;
        if (kk == 0) return;
        if (total <= k) {
            for (int e = tid; e < total; e += blockDim.x) o[e] = idxs[e];
            return;
        }
        uint32_t T; int teq;
        radix_threshold(keys, total, kk, sh, T, teq);
        ordered_compact(keys, total, T, teq, sh, [&](int pos, int e) { o[pos] = idxs[e]; });
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
