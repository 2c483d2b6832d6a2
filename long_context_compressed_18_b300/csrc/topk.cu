// Top-k selection ("DeepSeek V4 技术解读" §2.1: the Lightning Indexer keeps the
// k highest-scoring compressed entries per query).
//
// Exact selection on order-preserving 32-bit keys of the fp32 scores (-0
// folded onto +0): the k-th largest key T is found exactly (histogram levels
// over the keys, see radix_threshold, or one spread level plus a direct
// ranking of the boundary bin, see select_sparse), and the selection is every
// key > T plus the first (k - #{key > T}) elements equal to T in index order
// -- i.e. ranking by (score desc, index asc) -- written in ascending index
// order.  No floating-point atomics; the result does not depend on thread
// scheduling.
//
// Rows up to 16,384 entries take one CTA each with all keys in shared memory;
// rows up to TOPK_MAX_SINGLE take one fused CTA each (sampled threshold,
// collection, select); longer rows take two kernels (collect, select) over
// many CTAs, with the collection threshold from a sample of the row or, on
// the fused decode route, from the indexer's 32-entry maxima.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace csa {

constexpr int TOPK_THREADS = 512;
constexpr int TOPK_WARPS = TOPK_THREADS / 32;

// Scores are stored as fp32 or bf16 (ST); every load widens them to fp32
// exactly, so the keys -- and the selection -- are those of the stored values.
// at4 reads four consecutive scores (16 bytes of fp32, 8 of bf16) from a
// pointer aligned to their size (aligned4).
template <typename ST> struct ScoreIO;
template <> struct ScoreIO<float> {
    static __device__ __forceinline__ float at(const float* p, long long i) { return __ldg(p + i); }
    static __device__ __forceinline__ float4 at4(const float* p, long long i4)
    {
        return __ldg(reinterpret_cast<const float4*>(p) + i4);
    }
};
template <> struct ScoreIO<__nv_bfloat16> {
    static __device__ __forceinline__ float at(const __nv_bfloat16* p, long long i)
    {
        return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
    }
    static __device__ __forceinline__ float4 at4(const __nv_bfloat16* p, long long i4)
    {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p) + i4);
        return make_float4(bf16_bits_to_f32(u.x & 0xFFFFu), bf16_bits_to_f32(u.x >> 16),
                           bf16_bits_to_f32(u.y & 0xFFFFu), bf16_bits_to_f32(u.y >> 16));
    }
};
template <typename ST> __device__ __forceinline__ bool aligned4(const ST* p)
{
    return (reinterpret_cast<uintptr_t>(p) & (4 * sizeof(ST) - 1)) == 0;
}

// Radix levels over the 32-bit key: bits 31..21 (2048 bins), 20..10 (2048),
// 9..0 (1024).  The first level's histogram is built while the scores are
// loaded; the second while the elements of the selected first-level bin are
// compacted into a candidate list, so only that (short) list is scanned for
// the third level.  Rows whose selected bin overflows the list (heavy ties)
// scan the full key array instead.
constexpr int CAND_CAP = 2048;
constexpr int TOPK_SMEM_ROW = 16384;   // rows up to this length stage all their keys in shared memory

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
    // the earlier warps' totals, summed across the lanes
    uint32_t x = lane < warp ? sh.scan[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    uint32_t before = incl - tot + x;
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
                                int& take_eq_out, uint32_t* n_eq_out = nullptr)
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
    if (n_eq_out) *n_eq_out = sh.hist[sh.bin];   // keys equal to T
}

// Loads len fp32 scores into shared memory as keys and accumulates the
// first-level histogram.  Each thread keeps four 16-byte loads in flight
// (a whole 8,192-entry row in one batch), which keeps the kernel near the
// 32 registers of four CTAs an SM (a few spilled words cost less than the
// fourth CTA gains).
template <typename ST>
__device__ void load_score_keys(const ST* __restrict__ src, int len, uint32_t* keys, TopkShared& sh)
{
    const int tid = threadIdx.x;
    constexpr int U = 4;
    if (aligned4(src)) {
        const int n4 = len >> 2;
        for (int base = 0; base < n4; base += TOPK_THREADS * U) {
            float4 f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = base + u * TOPK_THREADS + tid;
                f[u] = v < n4 ? ScoreIO<ST>::at4(src, v) : make_float4(0.f, 0.f, 0.f, 0.f);
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
            const uint32_t key = score_key(ScoreIO<ST>::at(src, e));
            keys[e] = key;
            atomicAdd(&sh.hist[key >> 21], 1u);
        }
    } else {
        for (int base = 0; base < len; base += TOPK_THREADS * U) {
            float f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                f[u] = e < len ? ScoreIO<ST>::at(src, e) : 0.f;
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
template <typename Emit, typename Keys>
__device__ void ordered_compact_by(Keys keyat, int len, uint32_t T, int take_eq, TopkShared& sh, Emit emit)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (((len + TOPK_WARPS - 1) / TOPK_WARPS) + 31) & ~31;
    const int lo = min(len, warp * per), hi = min(len, lo + per);
    uint32_t n_take = 0, n_eq = 0;
    for (int e0 = lo; e0 < hi; e0 += 32) {
        const int e = e0 + lane;
        const uint32_t key = e < hi ? keyat(e) : 0u;
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
        const uint32_t key = e < hi ? keyat(e) : 0u;
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

template <typename Emit>
__device__ void ordered_compact(const uint32_t* keys, int len, uint32_t T, int take_eq, TopkShared& sh, Emit emit)
{
    ordered_compact_by([&](int e) { return keys[e]; }, len, T, take_eq, sh, emit);
}

// Rows of at most TOPK_SMEM_ROW entries: one CTA per row, the row's keys staged
// in shared memory, one radix select over them and an ordered compaction;
// writes the final indices, -1 padded.
template <typename ST>
__global__ void __launch_bounds__(TOPK_THREADS, 4) topk_smem_kernel(
    const ST* __restrict__ scores, long long ld, int n_q_rows, QPos qp, int m, int Nc,
    int k, int32_t* __restrict__ out, long long out_b_stride)
{
    grid_dep_entry();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ TopkShared sh;
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);
    const int r = (int)blockIdx.x;
    const int i = r % n_q_rows;   // query index within the chunk of rows
    const long long out_row = (long long)(r / n_q_rows) * out_b_stride + i;
    long long nvl = (qp.at(r / n_q_rows) + i + 1) / m;
    const int len = (int)(nvl < Nc ? nvl : Nc);
    const int tid = threadIdx.x;
    const int kk = min(k, len);
    int32_t* o = out + out_row * k;
    for (int p = kk + tid; p < k; p += TOPK_THREADS) o[p] = -1;
    if (kk == 0) return;
    if (len <= k) {
        for (int e = tid; e < len; e += TOPK_THREADS) o[e] = e;
        return;
    }
    clear_hist(sh, 2048);
    __syncthreads();
    load_score_keys(scores + (long long)r * ld, len, keys, sh);
    __syncthreads();
    uint32_t T;
    int teq;
    radix_threshold(keys, len, kk, sh, T, teq);
    ordered_compact(keys, len, T, teq, sh, [&](int pos, int e) { if (pos < kk) o[pos] = e; });
}

// ---------------------------------------------------------------------------
// Long rows (more than one CTA's capacity): the row counters are cleared (a
// memset, or the fused route's indexer), then two kernels.
//   collect  one CTA per 32768-entry chunk: every chunk CTA of a row derives
//            the same collection threshold thr -- from the keys of 4096
//            evenly spaced entries (a key at or below their key of rank
//            ~2k * 4096 / L plus a margin), or from the row's 32-entry maxima
//            written by the indexer (at or below the k-th largest maximum),
//            so expected to sit below the row's k-th largest key -- then
//            appends every entry of its chunk with key >= thr (with maxima:
//            reading only the 32-entry runs whose maximum reaches thr) to a
//            shared-memory list (4096 entries), whose slice of the row's
//            entry list is reserved with one global atomic;
//   select   one CTA per row: if the row collected at least k entries (so
//            the k-th largest key T is >= thr and every entry with key >= T
//            was collected) and no more than the list holds, T is found
//            exactly among the entries and the selected indices -- equal keys
//            taken in index order -- are written in ascending order
//            (select_sparse, or the bitmap route of select_entries for heavy
//            ties).  Otherwise (a threshold that misjudged the row) the row
//            is selected by the radix levels and ordered compaction streaming
//            the row from global memory.
// Both routes give the exact result; only their speed depends on the data.
// ---------------------------------------------------------------------------
constexpr int LR_CHUNK = 32768;
constexpr int LR_SAMPLES = 4096;
constexpr int LR_LOCAL_CAP = 4096;   // a chunk's shared-memory list (32 KB: four CTAs an SM)

static int lr_cap(int k) { return k * 4 > 8192 ? k * 4 : 8192; }

struct LongRowWs {
    uint32_t* cnt;    // [rows] entries collected (may exceed cap); cleared before the collection
    uint32_t* key;    // [rows][cap]
    int32_t* idx;     // [rows][cap]
    int cap;
};

static size_t lr_head_bytes(long long rows) { return ((size_t)rows * 4 + 255) / 256 * 256; }

static LongRowWs lr_ws(void* ws, long long rows, int k)
{
    LongRowWs w;
    uint8_t* p = reinterpret_cast<uint8_t*>(ws);
    w.cap = lr_cap(k);
    w.cnt = reinterpret_cast<uint32_t*>(p);
    p += lr_head_bytes(rows);
    w.key = reinterpret_cast<uint32_t*>(p);
    p += (size_t)rows * w.cap * 4;
    w.idx = reinterpret_cast<int32_t*>(p);
    return w;
}

__device__ __forceinline__ int visible_len(long long q_pos0, int i, int m, int Nc)
{
    const long long t1 = q_pos0 + i + 1;             // negative positions (a short sequence) see nothing
    const long long nvl = t1 > 0 ? t1 / m : 0;
    return (int)(nvl < Nc ? nvl : Nc);
}

// Streams score keys [c0, c0 + len) of a row: f(in_range, index, key) is
// called the same number of times in every lane (callers use warp ballots).
// 16-byte vector loads when the start is aligned, eight loads in flight.
template <typename ST, typename F>
__device__ __forceinline__ void stream_keys(const ST* __restrict__ row, int c0, int len, F f)
{
    constexpr int U = 8;
    const int tid = threadIdx.x;
    const ST* src = row + c0;
    int done = 0;
    if (aligned4(src)) {
        const int n4 = len >> 2;
        for (int base = 0; base < n4; base += TOPK_THREADS * U) {
            float4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e4 = base + u * TOPK_THREADS + tid;
                v[u] = e4 < n4 ? ScoreIO<ST>::at4(src, e4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e4 = base + u * TOPK_THREADS + tid;
                const bool in = e4 < n4;
                const int e = c0 + 4 * e4;
                f(in, e, score_key(v[u].x));
                f(in, e + 1, score_key(v[u].y));
                f(in, e + 2, score_key(v[u].z));
                f(in, e + 3, score_key(v[u].w));
            }
        }
        done = 4 * n4;
    }
    for (int base = done; base < len; base += TOPK_THREADS * U) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + u * TOPK_THREADS + tid;
            v[u] = e < len ? ScoreIO<ST>::at(src, e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + u * TOPK_THREADS + tid;
            f(e < len, c0 + e, score_key(v[u]));
        }
    }
}

// The float whose key is k (inverse of score_key on keys of non-NaN values).
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Collection threshold of a row: the keys of S = min(L, smax) entries in
// runs of 32 consecutive entries (whole cache lines), evenly spaced, ranked at
// t = 2 * kk * S / L + 8 (twice the expected rank of the k-th largest key,
// plus a margin).  The threshold only has to lie at or below the sample key
// of rank t.  When the samples' values span a finite, non-zero range, one
// 2,048-bin histogram linear in the value (a monotone map, so a higher bin
// never holds a smaller value) locates the bin holding rank t, and the
// smallest sample key in that bin is returned.  (Bins of the key are
// logarithmic in the value: across a sign change one is a quarter octave,
// far too coarse on its own.)  Otherwise the keys are spread as
// (key - lo) << s, s putting the top bit of hi - lo at bit 31, two histogram
// levels (bits 31..21, then 20..10 within the selected bin) locate rank t,
// and the lowest key whose spread key falls in that second-level bin is
// returned.  keys: shared buffer of smax entries.
template <int SMAX, typename ST>
__device__ uint32_t sample_threshold(const ST* __restrict__ row, int L, int kk, uint32_t* keys, TopkShared& sh)
{
    const int S = L < SMAX ? L : SMAX;
    const int runs = S / 32 > 0 ? S / 32 : 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    clear_hist(sh, 2048);
    constexpr int U = (SMAX + TOPK_THREADS - 1) / TOPK_THREADS;
    // run starts at run * (L - 32) / (runs - 1), in 24.8 fixed point: at most
    // (L - 32), so every sampled run lies inside the row
    const uint64_t step = ((uint64_t)(L > 32 ? L - 32 : 0) << 8) / (uint64_t)(runs > 1 ? runs - 1 : 1);
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int q = u * TOPK_THREADS + tid;
        const int run = q >> 5;
        const int e = (L < SMAX) ? q : (int)(((uint64_t)run * step) >> 8) + (q & 31);
        v[u] = q < S ? ScoreIO<ST>::at(row, e) : 0.f;
    }
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int q = u * TOPK_THREADS + tid;
        if (q < S) {
            const uint32_t key = score_key(v[u]);
            keys[q] = key;
            lo = min(lo, key);
            hi = max(hi, key);
        }
    }
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    if (lane == 0) {
        sh.scan[warp] = lo;
        sh.warp_take[warp] = hi;
    }
    __syncthreads();
    lo = lane < TOPK_WARPS ? sh.scan[lane] : 0xFFFFFFFFu;
    hi = lane < TOPK_WARPS ? sh.warp_take[lane] : 0u;
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    const long long want = 2ll * kk * S / L + 8;
    const int t_rank = (int)(want < S ? want : S);
    const float vlo = key_value(lo), vspan = key_value(hi) - vlo, vscale = 2048.f / vspan;
    if (isfinite(vspan) && vspan > 0.f && isfinite(vscale)) {
        auto vbin = [&](float x) { return min(2047, (int)((x - vlo) * vscale)); };
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (u * TOPK_THREADS + tid < S) atomicAdd(&sh.hist[vbin(v[u])], 1u);
        if (tid == 0) sh.n_cand = 0xFFFFFFFFu;   // the bin's smallest key
        __syncthreads();
        find_bin<2048>(sh, (uint32_t)t_rank);
        const int vb = (int)sh.bin;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int q = u * TOPK_THREADS + tid;
            if (q < S && vbin(v[u]) == vb) atomicMin(&sh.n_cand, keys[q]);
        }
        __syncthreads();
        const uint32_t T = sh.n_cand;
        __syncthreads();
        return T;
    }
    const uint32_t span = hi - lo;
    const int shl = span ? __clz(span) : 0;
    for (int q = tid; q < S; q += TOPK_THREADS) atomicAdd(&sh.hist[((keys[q] - lo) << shl) >> 21], 1u);
    __syncthreads();
    find_bin<2048>(sh, (uint32_t)t_rank);
    const uint32_t b1 = sh.bin, rem = (uint32_t)t_rank - sh.above;
    // second level: bits 20..10 of the spread keys in that bin
    clear_hist(sh, 2048);
    __syncthreads();
    for (int q = tid; q < S; q += TOPK_THREADS) {
        const uint32_t sk = (keys[q] - lo) << shl;
        if ((sk >> 21) == b1) atomicAdd(&sh.hist[(sk >> 10) & 0x7FFu], 1u);
    }
    __syncthreads();
    find_bin<2048>(sh, rem);
    // the lowest key whose spread key reaches the bin's: lo + ceil(sk / 2^shl)
    const uint64_t sk = ((uint64_t)b1 << 21) | ((uint64_t)sh.bin << 10);
    const uint32_t T = lo + (uint32_t)((sk + ((1ull << shl) - 1ull)) >> shl);
    __syncthreads();
    return T;
}


// Appends every entry e of [c0, c0 + len) of a row with key >= thr to the
// shared list (lkey, lidx) of capacity cap through the shared counter *n_loc;
// *n_loc counts every such entry, even past cap.  key >= thr is tested as the
// float comparison s >= value(thr), which orders -0 with +0 and never takes a
// NaN, exactly like the keys; a threshold key of 0 takes every entry.  Each
// thread builds a take mask over its batch of loads; one warp scan and one
// shared atomic per batch place the entries.
template <typename ST>
__device__ void collect_entries(const ST* __restrict__ row, int c0, int len, uint32_t thr, uint32_t* lkey,
                                int32_t* lidx, uint32_t cap, uint32_t* n_loc)
{
    const bool take_all = thr == 0u;
    const float tf = key_value(thr);
    const int tid = threadIdx.x, lane = tid & 31;
    const ST* src = row + c0;
    auto reserve = [&](uint32_t n) -> uint32_t {
        uint32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t wb = 0;
        if (lane == 31 && tot) wb = atomicAdd(n_loc, tot);
        wb = __shfl_sync(0xFFFFFFFFu, wb, 31);
        return wb + incl - n;
    };
    auto put = [&](uint32_t& pos, float v, int e) {
        if (pos < cap) {
            lkey[pos] = score_key(v);
            lidx[pos] = c0 + e;
        }
        ++pos;
    };
    constexpr int U = 8;
    int done = 0;
    if (aligned4(src)) {
        const int n4 = len >> 2;
        for (int base = 0; base < n4; base += TOPK_THREADS * U) {
            float4 f[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e4 = base + u * TOPK_THREADS + tid;
                f[u] = e4 < n4 ? ScoreIO<ST>::at4(src, e4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            uint32_t mask = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (base + u * TOPK_THREADS + tid < n4) {
                    mask |= (uint32_t)(take_all || f[u].x >= tf) << (4 * u);
                    mask |= (uint32_t)(take_all || f[u].y >= tf) << (4 * u + 1);
                    mask |= (uint32_t)(take_all || f[u].z >= tf) << (4 * u + 2);
                    mask |= (uint32_t)(take_all || f[u].w >= tf) << (4 * u + 3);
                }
            }
            if (!__any_sync(0xFFFFFFFFu, mask != 0u)) continue;
            uint32_t pos = reserve(__popc(mask));
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (mask & (0xFu << (4 * u))) {
                    const int e = 4 * (base + u * TOPK_THREADS + tid);
                    if (mask >> (4 * u) & 1u) put(pos, f[u].x, e);
                    if (mask >> (4 * u + 1) & 1u) put(pos, f[u].y, e + 1);
                    if (mask >> (4 * u + 2) & 1u) put(pos, f[u].z, e + 2);
                    if (mask >> (4 * u + 3) & 1u) put(pos, f[u].w, e + 3);
                }
            }
        }
        done = 4 * n4;
    }
    for (int base = done; base < len; base += TOPK_THREADS * U) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + u * TOPK_THREADS + tid;
            v[u] = e < len ? ScoreIO<ST>::at(src, e) : 0.f;
        }
        uint32_t mask = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * TOPK_THREADS + tid < len) mask |= (uint32_t)(take_all || v[u] >= tf) << u;
        if (!__any_sync(0xFFFFFFFFu, mask != 0u)) continue;
        uint32_t pos = reserve(__popc(mask));
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (mask >> u & 1u) put(pos, v[u], base + u * TOPK_THREADS + tid);
    }
}

// collect_entries restricted to the 32-entry runs of the chunk listed in
// runs[0..nr) (run j covers chunk entries 32 runs[j] .. 32 runs[j] + 31):
// the runs whose largest key (the indexer's warp maximum) reaches thr, the
// only ones that can hold an entry with key >= thr.  Eight lanes take a run,
// four consecutive entries each, and every lane issues its loads for U runs'
// worth before testing them.
template <typename ST>
__device__ void collect_runs(const ST* __restrict__ row, int c0, int len, uint32_t thr, const uint16_t* runs,
                             int nr, uint32_t* lkey, int32_t* lidx, uint32_t cap, uint32_t* n_loc)
{
    const bool take_all = thr == 0u;
    const float tf = key_value(thr);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const ST* src = row + c0;
    const bool vec = aligned4(src);
    constexpr int U = 4;   // run steps a lane loads at once (4 runs a warp a step)
    for (int j0 = warp * 4 * U; j0 < nr; j0 += TOPK_WARPS * 4 * U) {
        float v[U][4];
        int e0[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * 4 + (lane >> 3);
            e0[u] = j < nr ? 32 * (int)runs[j] + 4 * (lane & 7) : len;
            if (vec && e0[u] + 4 <= len) {
                const float4 f = ScoreIO<ST>::at4(src, e0[u] >> 2);
                v[u][0] = f.x; v[u][1] = f.y; v[u][2] = f.z; v[u][3] = f.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) v[u][q] = e0[u] + q < len ? ScoreIO<ST>::at(src, e0[u] + q) : 0.f;
            }
        }
        uint32_t mask = 0;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (e0[u] + q < len && (take_all || v[u][q] >= tf)) mask |= 1u << (4 * u + q);
        if (!__any_sync(0xFFFFFFFFu, mask != 0u)) continue;
        uint32_t incl = __popc(mask);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t wb = 0;
        if (lane == 31) wb = atomicAdd(n_loc, tot);
        uint32_t pos = __shfl_sync(0xFFFFFFFFu, wb, 31) + incl - __popc(mask);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (mask >> (4 * u + q) & 1u) {
                    if (pos < cap) {
                        lkey[pos] = score_key(v[u][q]);
                        lidx[pos] = c0 + e0[u] + q;
                    }
                    ++pos;
                }
    }
}

// Collection threshold from the row's warp maxima (wmax: the largest score
// key of each run of 32 consecutive entries, written by the indexer): a key
// at or below the kk-th largest of the nw = ceil(L / 32) maxima.  Those kk
// maxima are distinct entries, so at least kk entries have a key at or above
// it: every entry of the row's top kk does, and collecting key >= it is
// complete.  One histogram level suffices: the maxima crowd into a narrow
// key range, so they are spread first as (key - lo) << s (s putting the top
// bit of hi - lo at bit 31), and the returned key is the lower edge of the
// 2,048-bin level's bin holding rank kk (at most one bin, span / 2048, below
// the exact value).  With fewer maxima than kk, 0 (take every entry).
// keys: shared buffer of nw keys.
__device__ uint32_t wmax_threshold(const uint32_t* __restrict__ wrow, int nw, int kk, uint32_t* keys, TopkShared& sh)
{
    if (nw < kk) return 0u;
    const int tid = threadIdx.x;
    clear_hist(sh, 2048);
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    constexpr int WU = 16;   // loads in flight a thread
    for (int x0 = 0; x0 < nw; x0 += TOPK_THREADS * WU) {
        uint32_t v[WU];
#pragma unroll
        for (int u = 0; u < WU; ++u) {
            const int x = x0 + u * TOPK_THREADS + tid;
            v[u] = x < nw ? __ldcg(wrow + x) : 0u;
        }
#pragma unroll
        for (int u = 0; u < WU; ++u) {
            const int x = x0 + u * TOPK_THREADS + tid;
            if (x < nw) {
                keys[x] = v[u];
                lo = min(lo, v[u]);
                hi = max(hi, v[u]);
            }
        }
    }
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    if ((tid & 31) == 0) {
        sh.scan[tid >> 5] = lo;
        sh.warp_take[tid >> 5] = hi;
    }
    __syncthreads();
    lo = 0xFFFFFFFFu;
    hi = 0u;
    for (int q = 0; q < TOPK_WARPS; ++q) {
        lo = min(lo, sh.scan[q]);
        hi = max(hi, sh.warp_take[q]);
    }
    const uint32_t span = hi - lo;
    const int shl = span ? __clz(span) : 0;
    for (int x = tid; x < nw; x += TOPK_THREADS) atomicAdd(&sh.hist[((keys[x] - lo) << shl) >> 21], 1u);
    __syncthreads();
    find_bin<2048>(sh, (uint32_t)kk);
    return lo + ((sh.bin << 21) >> shl);
}

template <typename ST>
__global__ void __launch_bounds__(TOPK_THREADS, 2) topk_lr_collect_kernel(
    const ST* __restrict__ scores, long long ld, int n_q_rows, QPos qp, int m, int Nc, int k,
    int n_chunks, LongRowWs w, const uint32_t* __restrict__ wmax, int wmax_ld)
{
    grid_dep_entry();
    // the chunk's entries go to a shared-memory list, then one global atomic
    // reserves the chunk's slice of the row's list (whose order does not
    // matter to the select kernel)
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ uint32_t n_loc_s, base_s;
    __shared__ TopkShared sh;
    uint32_t* lkey = reinterpret_cast<uint32_t*>(smem_raw);   // [LR_LOCAL_CAP]
    int32_t* lidx = reinterpret_cast<int32_t*>(lkey + LR_LOCAL_CAP);
    const int r = blockIdx.x / n_chunks, c = blockIdx.x % n_chunks;
    const int L = visible_len(qp.at(r / n_q_rows), r % n_q_rows, m, Nc);
    if (L <= k) return;
    const int c0 = c * LR_CHUNK, len = max(0, min(LR_CHUNK, L - c0));
    if (len == 0) return;
    // every chunk CTA of the row derives the same threshold, from the row's
    // warp maxima when the indexer wrote them (and they fit the chunk list's
    // storage, which holds them meanwhile), else from the same samples
    static_assert(LR_LOCAL_CAP >= LR_SAMPLES, "sample keys live in the chunk list");
    const int nw = (L + 31) / 32;
    const bool by_runs = wmax && nw <= 2 * LR_LOCAL_CAP;
    const uint32_t thr = by_runs ? wmax_threshold(wmax + (long long)r * wmax_ld, nw, min(k, L), lkey, sh)
                                 : sample_threshold<LR_SAMPLES>(scores + (long long)r * ld, L, k, lkey, sh);
    __shared__ uint16_t runs_s[LR_CHUNK / 32];
    __shared__ uint32_t n_runs_s;
    if (threadIdx.x == 0) {
        n_loc_s = 0;
        n_runs_s = 0;
    }
    __syncthreads();
    const uint32_t cap = (uint32_t)w.cap;
    if (by_runs) {
        // the chunk's runs whose maximum (still in lkey) reaches thr; whole
        // warps take part in each ballot
        const int q0 = c0 / 32, nq = (len + 31) / 32, lane = threadIdx.x & 31;
        for (int t = threadIdx.x; t < ((nq + 31) & ~31); t += TOPK_THREADS) {
            const bool hit = t < nq && lkey[q0 + t] >= thr;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, hit);
            uint32_t p0 = 0;
            if (lane == 0 && bal) p0 = atomicAdd(&n_runs_s, (uint32_t)__popc(bal));
            p0 = __shfl_sync(0xFFFFFFFFu, p0, 0);
            if (hit) runs_s[p0 + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)t;
        }
        __syncthreads();
        collect_runs(scores + (long long)r * ld, c0, len, thr, runs_s, (int)n_runs_s, lkey, lidx, LR_LOCAL_CAP,
                     &n_loc_s);
    } else {
        collect_entries(scores + (long long)r * ld, c0, len, thr, lkey, lidx, LR_LOCAL_CAP, &n_loc_s);
    }
    __syncthreads();
    const uint32_t n_all = n_loc_s;
    // counts every entry, even past the row's capacity; a chunk that
    // overflowed its own list pushes the count past it too, so the row is
    // selected by the streamed route
    if (threadIdx.x == 0)
        base_s = atomicAdd(w.cnt + r, n_all + (n_all > (uint32_t)LR_LOCAL_CAP ? cap + 1u : 0u));
    __syncthreads();
    const uint32_t base = base_s, n_loc = min(n_all, (uint32_t)LR_LOCAL_CAP);
    uint32_t* ek = w.key + (size_t)r * cap;
    int32_t* ei = w.idx + (size_t)r * cap;
    for (uint32_t q = threadIdx.x; q < n_loc; q += TOPK_THREADS) {
        if (base + q < cap) {
            ek[base + q] = lkey[q];
            ei[base + q] = lidx[q];
        }
    }
}

// Words of one index bitmap of a row of L entries, rounded up to whole
// 16-byte groups.
__host__ __device__ constexpr int bitmap_words(int L) { return (((L + 31) / 32) + 3) & ~3; }

// Exact selection among a row's entries (ekey, eidx: n entries in shared
// memory, every entry of the row whose key is at least some threshold,
// n >= kk) -- the top kk by (score desc, index asc) -- written to o in
// ascending index order.  bitmaps: shared memory for two bitmaps of
// bitmap_words(L) words each (16-byte aligned).
__device__ void select_entries(uint32_t* ekey, const int32_t* eidx, int n, int kk, int L, uint32_t* bitmaps,
                               TopkShared& sh, int32_t* __restrict__ o)
{
    const int tid = threadIdx.x;
    const int nw = (L + 31) / 32, nw4 = bitmap_words(L);
    uint32_t* sel = bitmaps;
    uint32_t* eqm = bitmaps + nw4;
    clear_hist(sh, 2048);
    for (int x = tid; x < 2 * nw4; x += TOPK_THREADS) bitmaps[x] = 0u;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int e = tid; e < n; e += TOPK_THREADS) {
        lo = min(lo, ekey[e]);
        hi = max(hi, ekey[e]);
    }
    // Raw keys crowd into a few first-level bins; rank the entries instead by
    // (key - lo) << s, s putting the top bit of hi - lo at bit 31 -- strictly
    // increasing in key, so the threshold and the ties (and hence the
    // selection) are the same, and the first radix level spreads over all
    // its bins.
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    if ((tid & 31) == 0) {
        sh.scan[tid >> 5] = lo;
        sh.warp_take[tid >> 5] = hi;
    }
    __syncthreads();
    lo = 0xFFFFFFFFu;
    hi = 0u;
    for (int q = 0; q < TOPK_WARPS; ++q) {
        lo = min(lo, sh.scan[q]);
        hi = max(hi, sh.warp_take[q]);
    }
    const uint32_t span = hi - lo;
    const int shl = span ? __clz(span) : 0;
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const uint32_t tk = (ekey[e] - lo) << shl;
        ekey[e] = tk;
        atomicAdd(&sh.hist[tk >> 21], 1u);
    }
    __syncthreads();
    uint32_t T, n_eq;
    int teq;
    radix_threshold(ekey, n, kk, sh, T, teq, &n_eq);
    __syncthreads();
    // mark the selection; keys equal to T join it directly unless only some
    // of them are taken (then the first teq in index order, below)
    const bool all_eq = n_eq == (uint32_t)teq;
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const uint32_t key = ekey[e];
        const int j = eidx[e];
        if (j < 0 || j >= L) continue;
        if (key > T || (key == T && all_eq)) atomicOr(&sel[j >> 5], 1u << (j & 31));
        else if (key == T) atomicOr(&eqm[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    if (!all_eq) {
        // warp-cooperative walk of the tie bitmap: warp w owns words [wa, wb)
        const int per_w = ((nw + TOPK_WARPS - 1) / TOPK_WARPS + 31) & ~31;
        const int wa = min(nw, warp * per_w), wb = min(nw, wa + per_w);
        uint32_t t = 0;
        for (int x = wa + lane; x < wb; x += 32) t += __popc(eqm[x]);
#pragma unroll
        for (int dd = 16; dd > 0; dd >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, dd);
        if (lane == 0) sh.scan[warp] = t;
        __syncthreads();
        uint32_t rank = 0;
        for (int q = 0; q < warp; ++q) rank += sh.scan[q];
        for (int x0 = wa; x0 < wb; x0 += 32) {
            const int x = x0 + lane;
            uint32_t bits = x < wb ? eqm[x] : 0u;
            const uint32_t nb = __popc(bits);
            uint32_t incl = nb;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, dd);
                if (lane >= dd) incl += v;
            }
            const uint32_t r0 = rank + incl - nb;
            if (bits) {
                if (r0 + nb <= (uint32_t)teq) {
                    sel[x] |= bits;
                } else if (r0 < (uint32_t)teq) {
                    for (uint32_t q = r0; q < (uint32_t)teq; ++q) {
                        const uint32_t low = bits & (0u - bits);
                        sel[x] |= low;
                        bits ^= low;
                    }
                }
            }
            rank += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        __syncthreads();
    }
    // output slot of index j: (selected indices in words before j's) +
    // (selected bits below j in its word); the per-word prefix goes into
    // the tie bitmap's storage.  Warp w owns words [wa, wb): its lanes read
    // consecutive words (no bank conflicts) and a warp scan carries the count.
    uint32_t* wpre = eqm;
    {
        const int nq = nw4 / 4;   // 16-byte groups of words; a lane takes one group a step
        const int per_w = ((nq + TOPK_WARPS - 1) / TOPK_WARPS + 31) & ~31;
        const int qa = min(nq, warp * per_w), qb = min(nq, qa + per_w);
        const uint4* sel4 = reinterpret_cast<const uint4*>(sel);
        uint4* wpre4 = reinterpret_cast<uint4*>(wpre);
        uint32_t t = 0;
        for (int q = qa + lane; q < qb; q += 32) {
            const uint4 w4 = sel4[q];
            t += __popc(w4.x) + __popc(w4.y) + __popc(w4.z) + __popc(w4.w);
        }
#pragma unroll
        for (int dd = 16; dd > 0; dd >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, dd);
        if (lane == 0) sh.scan[warp] = t;
        __syncthreads();
        uint32_t run = 0;
        for (int q = 0; q < warp; ++q) run += sh.scan[q];
        for (int q0 = qa; q0 < qb; q0 += 32) {
            const int q = q0 + lane;
            const uint4 w4 = q < qb ? sel4[q] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t c0 = __popc(w4.x), c1 = __popc(w4.y), c2 = __popc(w4.z), c3 = __popc(w4.w);
            const uint32_t c = c0 + c1 + c2 + c3;
            uint32_t incl = c;
#pragma unroll
            for (int dd = 1; dd < 32; dd <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, dd);
                if (lane >= dd) incl += v;
            }
            const uint32_t b0 = run + incl - c;
            if (q < qb) wpre4[q] = make_uint4(b0, b0 + c0, b0 + c0 + c1, b0 + c0 + c1 + c2);
            run += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
    }
    __syncthreads();
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const int j = eidx[e];
        if (j < 0 || j >= L) continue;
        const uint32_t word = sel[j >> 5], bit = 1u << (j & 31);
        if (word & bit) {
            const uint32_t pos = wpre[j >> 5] + __popc(word & (bit - 1u));
            if (pos < (uint32_t)kk) o[pos] = j;
        }
    }
}

// Exact selection of a row's top kk streamed from global memory: the three
// radix levels, then the ordered compaction.
template <typename ST>
__device__ void select_streaming(const ST* __restrict__ row, int L, int kk, TopkShared& sh,
                                 int32_t* __restrict__ o)
{
    clear_hist(sh, 2048);
    __syncthreads();
    stream_keys(row, 0, L, [&](bool in, int, uint32_t key) {
        if (in) atomicAdd(&sh.hist[key >> 21], 1u);
    });
    __syncthreads();
    find_bin<2048>(sh, (uint32_t)kk);
    const uint32_t b1 = sh.bin;
    uint32_t rem = (uint32_t)kk - sh.above;
    clear_hist(sh, 2048);
    __syncthreads();
    stream_keys(row, 0, L, [&](bool in, int, uint32_t key) {
        if (in && (key >> 21) == b1) atomicAdd(&sh.hist[(key >> 10) & 0x7FFu], 1u);
    });
    __syncthreads();
    find_bin<2048>(sh, rem);
    const uint32_t pre = (b1 << 11) | sh.bin;
    rem -= sh.above;
    clear_hist(sh, 1024);
    __syncthreads();
    stream_keys(row, 0, L, [&](bool in, int, uint32_t key) {
        if (in && (key >> 10) == pre) atomicAdd(&sh.hist[key & 0x3FFu], 1u);
    });
    __syncthreads();
    find_bin<1024>(sh, rem);
    const uint32_t T = (pre << 10) | sh.bin;
    const int teq = (int)(rem - sh.above);
    ordered_compact_by([&](int e) { return score_key(ScoreIO<ST>::at(row, e)); }, L, T, teq, sh,
                       [&](int pos, int e) { if (pos < kk) o[pos] = e; });
}

// Words of select_sparse's scratch: the 2,048 bucket starts, then kk slots.
__host__ __device__ constexpr int sparse_scratch_words(int k) { return 2048 + ((k + 3) & ~3); }

// Exact selection for an entry list much shorter than its row (ekey, eidx: n
// entries in shared memory, every entry of the row whose key is at least
// some threshold, n >= kk; L <= 2^20), in steps sized by the list, not by
// the row:
//   1. the keys are spread as (key - lo) << s (strictly increasing) and
//      counted in a 2,048-bin histogram; the bin b holding rank kk is found;
//   2. the entries of bin b (usually a handful) are ranked among themselves
//      by direct comparison, which gives the kk-th largest key T exactly;
//   3. the kk entries with key >= T are counted into 2,048 buckets of
//      consecutive indices (j >> shift), the bucket starts found by a prefix
//      sum, and each entry scattered into its bucket; each one's slot is then
//      its bucket start plus the number of its bucket's entries with a
//      smaller index, so the output is in ascending index order.
// Returns false, before writing o, when the list needs the general route
// (select_entries): bin b holds more entries than the CTA has threads, or
// only some of the entries equal to T are taken (index order among ties).
// scratch: sparse_scratch_words(kk) words of shared memory.  lo_t / hi_t:
// this thread's minimum / maximum over the keys it wrote to ekey, when the
// caller tracked them (have_range), else the keys are scanned here.
__device__ bool select_sparse(uint32_t* ekey, const int32_t* eidx, int n, int kk, int L, uint32_t* scratch,
                              TopkShared& sh, int32_t* __restrict__ o, bool have_range = false,
                              uint32_t lo_t = 0xFFFFFFFFu, uint32_t hi_t = 0u)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    clear_hist(sh, 2048);
    if (tid == 0) sh.n_cand = 0;
    uint32_t lo = lo_t, hi = hi_t;
    if (!have_range) {
        for (int e = tid; e < n; e += TOPK_THREADS) {
            lo = min(lo, ekey[e]);
            hi = max(hi, ekey[e]);
        }
    }
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    if (lane == 0) {
        sh.scan[warp] = lo;
        sh.warp_take[warp] = hi;
    }
    __syncthreads();
    lo = lane < TOPK_WARPS ? sh.scan[lane] : 0xFFFFFFFFu;
    hi = lane < TOPK_WARPS ? sh.warp_take[lane] : 0u;
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, dd));
        hi = max(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, dd));
    }
    const uint32_t span = hi - lo;
    const int shl = span ? __clz(span) : 0;
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const uint32_t tk = (ekey[e] - lo) << shl;
        ekey[e] = tk;
        atomicAdd(&sh.hist[tk >> 21], 1u);
    }
    __syncthreads();
    // 1. the bin of rank kk; rem = kk's rank within it
    find_bin<2048>(sh, (uint32_t)kk);
    const uint32_t b1 = sh.bin, rem = (uint32_t)kk - sh.above;
    // the bin's entries (their order is irrelevant); usually a handful, so
    // each one reserves its own slot
    if (tid == 0) sh.warp_eq[0] = 0xFFFFFFFFu;   // no T found yet
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const uint32_t key = ekey[e];
        if ((key >> 21) == b1) {
            const uint32_t pos = atomicAdd(&sh.n_cand, 1u);
            if (pos < CAND_CAP) sh.cand[pos] = key;
        }
    }
    __syncthreads();
    const int nc = (int)sh.n_cand;
    if (nc > TOPK_THREADS) return false;
    // 2. T: the candidate with gt < rem <= gt + eq (every thread holding a
    // key equal to T writes the same values)
    if (tid < nc) {
        const uint32_t kt = sh.cand[tid];
        uint32_t gt = 0, eq = 0;
        for (int c = 0; c < nc; ++c) {
            const uint32_t kc = sh.cand[c];
            gt += kc > kt;
            eq += kc == kt;
        }
        if (gt < rem && rem <= gt + eq) {
            sh.bin = kt;
            sh.above = rem - gt;   // taken among the keys equal to T
            sh.warp_eq[0] = eq;    // keys equal to T
        }
    }
    __syncthreads();
    const uint32_t T = sh.bin;
    if (sh.above != sh.warp_eq[0]) return false;
    // 3. ascending index order by bucket counting
    const int bits = L > 1 ? 32 - __clz((uint32_t)(L - 1)) : 1;
    const int shift = bits > 11 ? bits - 11 : 0;
    uint32_t* start = scratch;        // [2048]
    int32_t* slot = reinterpret_cast<int32_t*>(scratch + 2048);   // [kk]
    __syncthreads();                  // every thread has read sh.bin / sh.above
    clear_hist(sh, 2048);
    __syncthreads();
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const int j = eidx[e];
        if (ekey[e] >= T && (unsigned)j < (unsigned)L) atomicAdd(&sh.hist[j >> shift], 1u);
    }
    __syncthreads();
    {
        constexpr int BPT = 2048 / TOPK_THREADS;
        uint32_t c[BPT], tot = 0;
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            c[q] = sh.hist[tid * BPT + q];
            tot += c[q];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
            const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
            if (lane >= o2) incl += t;
        }
        if (lane == 31) sh.scan[warp] = incl;
        __syncthreads();
        uint32_t x = lane < warp ? sh.scan[lane] : 0u;
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o2);
        uint32_t run = x + incl - tot;
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            start[tid * BPT + q] = run;
            sh.hist[tid * BPT + q] = run;   // the bucket's fill cursor
            run += c[q];
        }
        if (tid == TOPK_THREADS - 1) sh.n_cand = run;   // entries taken
    }
    __syncthreads();
    if (sh.n_cand != (uint32_t)kk) return false;   // cannot happen for a valid list
    for (int e = tid; e < n; e += TOPK_THREADS) {
        const int j = eidx[e];
        if (ekey[e] >= T && (unsigned)j < (unsigned)L) {
            const uint32_t p = atomicAdd(&sh.hist[j >> shift], 1u);
            if (p < (uint32_t)kk) slot[p] = j;
        }
    }
    __syncthreads();
    for (int q = tid; q < kk; q += TOPK_THREADS) {
        const int j = slot[q];
        const int b = j >> shift;
        const uint32_t st = start[b], en = min(sh.hist[b], (uint32_t)kk);
        uint32_t r = 0;
        for (uint32_t i = st; i < en; ++i) r += slot[i] < j;
        o[st + r] = j;
    }
    return true;
}

template <typename ST>
__global__ void __launch_bounds__(TOPK_THREADS) topk_lr_select_kernel(
    const ST* __restrict__ scores, long long ld, int n_q_rows, QPos qp, int m, int Nc, int k,
    LongRowWs w, int fast_ok, int32_t* __restrict__ out, long long out_b_stride)
{
    grid_dep_entry();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ TopkShared sh;
    const int r = blockIdx.x;
    const int i = r % n_q_rows;
    int32_t* o = out + ((long long)(r / n_q_rows) * out_b_stride + i) * k;
    const int L = visible_len(qp.at(r / n_q_rows), i, m, Nc);
    const int kk = min(k, L);
    const int tid = threadIdx.x;
    for (int p = kk + tid; p < k; p += TOPK_THREADS) o[p] = -1;
    if (kk == 0) return;
    if (L <= k) {
        for (int e = tid; e < L; e += TOPK_THREADS) o[e] = e;
        return;
    }
    const ST* row = scores + (long long)r * ld;
    // the list's first TOPK_THREADS * 8 slots are loaded together with its
    // count (slots past the count hold stale words and are dropped; the list
    // has at least that many slots), saving a round trip
    static_assert(TOPK_THREADS * 8 <= 8192, "the first batch lies inside the row's list");
    uint32_t kv[8];
    int32_t iv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        kv[u] = __ldcg(w.key + (size_t)r * w.cap + u * TOPK_THREADS + tid);
        iv[u] = __ldcg(w.idx + (size_t)r * w.cap + u * TOPK_THREADS + tid);
    }
    const uint32_t got = __ldcg(w.cnt + r);
    if (fast_ok && got >= (uint32_t)kk && got <= (uint32_t)w.cap) {
        // two bitmaps of the row (or select_sparse's scratch), then the list
        uint32_t* bitmaps = reinterpret_cast<uint32_t*>(smem_raw);
        uint32_t* ekey = bitmaps + max(2 * bitmap_words(L), sparse_scratch_words(k));   // [cap]
        int32_t* eidx = reinterpret_cast<int32_t*>(ekey + w.cap);
        const int n = (int)got;
        uint32_t lo = 0xFFFFFFFFu, hi = 0u;
        for (int base = 0; base < n; base += TOPK_THREADS * 8) {
            if (base > 0) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = base + u * TOPK_THREADS + tid;
                    kv[u] = e < n ? __ldcg(w.key + (size_t)r * w.cap + e) : 0u;
                    iv[u] = e < n ? __ldcg(w.idx + (size_t)r * w.cap + e) : 0;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = base + u * TOPK_THREADS + tid;
                if (e < n) {
                    ekey[e] = kv[u];
                    eidx[e] = iv[u];
                    lo = min(lo, kv[u]);
                    hi = max(hi, kv[u]);
                }
            }
        }
        __syncthreads();
        if (!select_sparse(ekey, eidx, n, kk, L, bitmaps, sh, o, true, lo, hi)) {
            __syncthreads();
            select_entries(ekey, eidx, n, kk, L, bitmaps, sh, o);
        }
        return;
    }
    select_streaming(row, L, kk, sh, o);
}

// ---------------------------------------------------------------------------
// Rows of at most TOPK_MAX_SINGLE entries: one CTA per row runs the same
// steps as the long-row kernels, fused -- a sampled threshold (or the whole
// row when it fits the entry list), one collection pass into shared memory,
// the exact select over the entries -- with the streamed route for rows whose
// sample misjudges them.  About 57 KB of shared memory at k = 1024 and at most
// 64 registers a thread, so two rows run per SM.
// ---------------------------------------------------------------------------
constexpr int ROW_SAMPLES = 2048;

// Entry-list capacity of the fused kernel: enough for about twice k
// collected entries (rows that fit take everything, no sampling).
static int row_cap(int N_c, int k)
{
    (void)N_c;
    return 2 * k + 2048 > 4096 ? 2 * k + 2048 : 4096;
}

static size_t row_smem_bytes(int N_c, int k)
{
    return (size_t)row_cap(N_c, k) * 8 + (size_t)std::max(2 * bitmap_words(N_c), sparse_scratch_words(k)) * 4;
}

template <typename ST>
__global__ void __launch_bounds__(TOPK_THREADS, 2) topk_kernel(
    const ST* __restrict__ scores, long long ld, int n_q_rows, QPos qp, int m, int Nc, int k, int cap,
    int32_t* __restrict__ out, long long out_b_stride)
{
    grid_dep_entry();
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ TopkShared sh;
    __shared__ uint32_t n_cnt;
    uint32_t* ekey = reinterpret_cast<uint32_t*>(smem_raw);   // [cap]; holds the samples first
    int32_t* eidx = reinterpret_cast<int32_t*>(ekey + cap);   // [cap]
    uint32_t* bitmaps = reinterpret_cast<uint32_t*>(eidx + cap);
    const int r = (int)blockIdx.x;
    const int i = r % n_q_rows;   // query index within the chunk of rows
    int32_t* o = out + ((long long)(r / n_q_rows) * out_b_stride + i) * k;
    const int L = visible_len(qp.at(r / n_q_rows), i, m, Nc);
    const int kk = min(k, L);
    const int tid = threadIdx.x;
    for (int p = kk + tid; p < k; p += TOPK_THREADS) o[p] = -1;
    if (kk == 0) return;
    if (L <= k) {
        for (int e = tid; e < L; e += TOPK_THREADS) o[e] = e;
        return;
    }
    const ST* row = scores + (long long)r * ld;
    const uint32_t thr = L > cap ? sample_threshold<ROW_SAMPLES>(row, L, kk, ekey, sh) : 0u;   // 0: take all
    if (tid == 0) n_cnt = 0;
    __syncthreads();
    collect_entries(row, 0, L, thr, ekey, eidx, (uint32_t)cap, &n_cnt);
    __syncthreads();
    const uint32_t n = n_cnt;
    if (n >= (uint32_t)kk && n <= (uint32_t)cap) {
        if (!select_sparse(ekey, eidx, (int)n, kk, L, bitmaps, sh, o)) {
            __syncthreads();
            select_entries(ekey, eidx, (int)n, kk, L, bitmaps, sh, o);
        }
        return;
    }
    select_streaming(row, L, kk, sh, o);
}

// Chunking plan shared by the launcher and the workspace query.
TopkPlan topk_plan(int N_c, int k)
{
    TopkPlan p;
    (void)k;
    if (N_c <= TOPK_MAX_SINGLE) {
        p.chunk = N_c > 0 ? N_c : 1;
        p.n_chunks = 1;
    } else {
        p.chunk = LR_CHUNK;
        p.n_chunks = (N_c + LR_CHUNK - 1) / LR_CHUNK;
    }
    return p;
}

bool topk_supported(int N_c, int k) { return k >= 1 && k <= 4096 && N_c >= 0 && N_c <= TOPK_MAX_ROW; }

bool topk_rows_ok(long long rows, int N_c, int k)
{
    // one CTA per row (times the chunks of a long row) in grid.x
    const TopkPlan p = topk_plan(N_c, k);
    return rows >= 0 && rows * p.n_chunks <= (long long)INT_MAX;
}

size_t topk_workspace_bytes(long long rows, int N_c, int k)
{
    TopkPlan p = topk_plan(N_c, k);
    if (p.n_chunks == 1 || rows <= 0) return 0;
    return lr_head_bytes(rows) + (size_t)rows * lr_cap(k) * 8;
}

// The select kernel over a row's entry list.  The fast route needs two
// bitmaps of the row and the entry list in shared memory; shapes beyond that
// stream every row instead.
template <typename ST>
static cudaError_t launch_select(const ST* scores, long long ld, int n_q_rows, QPos q_pos0, int m, int N_c,
                                 int k, const LongRowWs& w, int rows, int32_t* out, long long out_b_stride,
                                 cudaStream_t s)
{
    size_t smem = (size_t)std::max(2 * bitmap_words(N_c), sparse_scratch_words(k)) * 4 + (size_t)w.cap * 8;
    const int fast_ok = smem <= (size_t)200 * 1024;
    if (!fast_ok) smem = 0;
    auto kern = topk_lr_select_kernel<ST>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_pdl(kern, dim3(rows), dim3(TOPK_THREADS), smem, s, scores, ld, n_q_rows, q_pos0, m, N_c, k, w, fast_ok, out, out_b_stride);
    return cudaGetLastError();
}

template <typename ST>
static cudaError_t launch_topk_t(const ST* scores, long long ld, int B, int n_q_rows, QPos q_pos0, int m,
                                 int N_c, int k, int32_t* out, long long out_b_stride, void* ws, cudaStream_t s,
                                 const uint32_t* wmax, int wmax_ld, bool counters_clear)
{
    const long long rows_ll = (long long)B * n_q_rows;
    if (rows_ll == 0) return cudaSuccess;
    if (!topk_rows_ok(rows_ll, N_c, k)) return cudaErrorInvalidConfiguration;   // callers check first
    const int rows = (int)rows_ll;
    TopkPlan p = topk_plan(N_c, k);
    if (p.n_chunks == 1 && N_c <= TOPK_SMEM_ROW) {
        const size_t smem = (size_t)(N_c > 0 ? N_c : 1) * sizeof(uint32_t);
        auto kern = topk_smem_kernel<ST>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        (void)launch_pdl(kern, dim3(rows), dim3(TOPK_THREADS), smem, s, scores, ld, n_q_rows, q_pos0, m, N_c, k, out, out_b_stride);
        return cudaGetLastError();
    }
    if (p.n_chunks == 1) {
        const size_t smem = row_smem_bytes(N_c, k);
        auto kern = topk_kernel<ST>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        (void)launch_pdl(kern, dim3(rows), dim3(TOPK_THREADS), smem, s, scores, ld, n_q_rows, q_pos0, m, N_c, k, row_cap(N_c, k), out, out_b_stride);
        return cudaGetLastError();
    }
    const LongRowWs w = lr_ws(ws, rows, k);
    if (!counters_clear) {
        cudaError_t e = cudaMemsetAsync(w.cnt, 0, (size_t)rows * sizeof(uint32_t), s);
        if (e != cudaSuccess) return e;
    }
    const size_t csmem = (size_t)LR_LOCAL_CAP * 8;
    auto ckern = topk_lr_collect_kernel<ST>;
    cudaFuncSetAttribute(ckern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
    (void)launch_pdl(ckern, dim3(rows * p.n_chunks), dim3(TOPK_THREADS), csmem, s, scores, ld, n_q_rows, q_pos0, m, N_c, k, p.n_chunks, w, wmax, wmax_ld);
    return launch_select(scores, ld, n_q_rows, q_pos0, m, N_c, k, w, rows, out, out_b_stride, s);
}

cudaError_t launch_topk(const void* scores, bool scores_bf16, long long ld, int B, int n_q_rows, QPos q_pos0,
                        int m, int N_c, int k, int32_t* out, long long out_b_stride, void* ws,
                        cudaStream_t s, const uint32_t* wmax, int wmax_ld, bool counters_clear)
{
    if (scores_bf16)
        return launch_topk_t(reinterpret_cast<const __nv_bfloat16*>(scores), ld, B, n_q_rows, q_pos0, m, N_c, k, out,
                             out_b_stride, ws, s, wmax, wmax_ld, counters_clear);
    return launch_topk_t(reinterpret_cast<const float*>(scores), ld, B, n_q_rows, q_pos0, m, N_c, k, out,
                         out_b_stride, ws, s, wmax, wmax_ld, counters_clear);
}

uint32_t* topk_row_counters(void* ws) { return reinterpret_cast<uint32_t*>(ws); }

bool topk_long_rows(int N_c, int k) { return topk_plan(N_c, k).n_chunks > 1; }

int topk_wmax_ld(int N_c) { return (N_c + 31) / 32; }

size_t topk_wmax_bytes(long long rows, int N_c)
{
    return ((size_t)rows * topk_wmax_ld(N_c) * 4 + 255) / 256 * 256;
}

}  // namespace csa
