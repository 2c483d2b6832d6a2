// Lightning Indexer scores ("DeepSeek V4 技术解读" §2.1: indexer queries of 64
// heads x 128 dims are scored against the compressed entries; §五: the QK path
// runs in FP8/FP4).
//
//     s(t, j) = sk(j) * sum_h sq(t, h) * <q(t, h), k(j)>      for j < nv(t)
//
// tcgen05 kernel (BF16 x BF16 via kind::f16, E4M3 x E4M3 via kind::f8f6f4,
// fp32 accumulation in tensor memory).  The contraction is laid out with the
// keys on the MMA's M side and (token, head) pairs on its N side:
//     D[128 keys, T*64] = K_tile[128 x 128] * Q_group[T*64 x 128]^T
// so that each TMEM lane holds one key and the head sum of the epilogue is a
// per-thread reduction over 64 columns (no cross-lane traffic).  T = 4 tokens
// (N = 256) for prefill, T = 1 (N = 64) for decode.
//
// Warp roles: warp 0 issues TMA loads (the query group once, then a ring of
// key tiles); warp 1 owns the TMEM allocation and issues the MMAs from one
// thread; 4 * T epilogue warps (one token each, four per TMEM lane quadrant
// for T = 4) drain TMEM (tcgen05.ld), apply the scales, sum over heads and
// store fp32 scores.
//
// FP4 key cache at decode (KFP4, T = 1): warp 0 streams the packed E2M1 tiles
// (64 bytes a key) into a ring of raw stages, and eight converter warps widen
// them to E4M3 in the swizzled operand layout the MMA reads -- the §五
// FP4 -> FP8 step inside the kernel, so the keys cross HBM once at half a
// byte an element.  The widening is the one of fp4_to_e4m3_kernel below
// (row scale S = 2^(floor(log2 max_b sc_b) - 5), x8 = E4M3(e sc_b / S)),
// done per 32-element block through a 16-entry byte table: the block's eight
// magnitudes E4M3(|e| sc_b / S) are computed once, each code's magnitude bits
// pick its byte with a byte permute, and its sign bit flips the result's.
// The epilogue recomputes S from the key's four block scales.  Accumulators are multi-buffered in
// TMEM so the MMA of tile i+1 overlaps the epilogue of tile i.  Every mbarrier
// wait is bounded; on a timeout the CTA drains its copies and MMAs, frees
// TMEM and exits with the device status word set.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace idx {
// warps 0-1 producer and MMA issuer, then the epilogue warps, one token each:
// 4 for one token per group (decode), 16 for four tokens (four warps per TMEM
// lane quadrant, so each scheduler has four epilogue warps to switch between)
template <int T> constexpr int epi_warps() { return 4 * T; }
constexpr int CONV_WARPS = 4;     // FP4 -> E4M3 converter warps (KFP4)
template <int T, bool KFP4 = false> constexpr int threads() { return 64 + 32 * (epi_warps<T>() + (KFP4 ? CONV_WARPS : 0)); }
constexpr int BLOCK_KEYS = 128;   // MMA M
constexpr int CONV_ITEMS = BLOCK_KEYS * 4 / (32 * CONV_WARPS);   // 32-element blocks a converter thread a tile
constexpr int SC_DEPTH = 4;       // tiles of key scales in flight (decode groups)
constexpr int HEADS = 64;         // indexer heads
constexpr int DIM = 128;          // indexer head dim
constexpr int ATOM_BYTES_ROW = 128;

template <bool FP8, int T, bool KFP4 = false> struct Cfg {
    static constexpr int N = HEADS * T;
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ATOMS = DIM * ELEM / ATOM_BYTES_ROW;  // 128-byte K-major column blocks
    static constexpr int KSTEP_ELEMS = FP8 ? 32 : 16;          // K per MMA instruction
    static constexpr int KSTEPS = DIM / KSTEP_ELEMS;
    static constexpr int KSTEPS_PER_ATOM = KSTEPS / ATOMS;
    static constexpr int Q_ATOM = N * ATOM_BYTES_ROW;
    static constexpr int Q_BYTES = Q_ATOM * ATOMS;
    static constexpr int K_ATOM = BLOCK_KEYS * ATOM_BYTES_ROW;
    static constexpr int K_BYTES = K_ATOM * ATOMS;
    static constexpr int STAGES = KFP4 ? 4 : (T == 1) ? 6 : (FP8 ? 6 : 4);
    static constexpr int ACC = (T == 1) ? 4 : 2;
    static constexpr int TMEM_COLS = ACC * N;   // 256 or 512
    static constexpr uint32_t IDESC = instr_desc(FP8 ? 0u : 1u, FP8 ? 0u : 1u, BLOCK_KEYS, N);
    // packed E2M1 key tiles (KFP4): 64 bytes a key
    static constexpr int RAW_STAGES = KFP4 ? 3 : 0;
    static constexpr int RAW_BYTES = BLOCK_KEYS * DIM / 2;
    // rings of key scales copied ahead with cp.async (decode groups): one
    // word a key for each epilogue thread, CONV_ITEMS words for each converter
    static constexpr bool SC_RING = (T == 1);
    static constexpr int E_RING = SC_RING ? SC_DEPTH * 32 * epi_warps<T>() * 4 : 0;
    static constexpr int C_RING = KFP4 ? SC_DEPTH * 32 * CONV_WARPS * CONV_ITEMS * 4 : 0;
    // barriers: full[STAGES], empty[STAGES], acc_full[ACC], acc_empty[ACC], q, mma_done,
    // raw_full[RAW_STAGES], raw_empty[RAW_STAGES]
    static constexpr int N_BARS = 2 * STAGES + 2 * ACC + 2 + 2 * RAW_STAGES;
    static constexpr int SMEM = 1024 /*align slack*/ + Q_BYTES + STAGES * K_BYTES + RAW_STAGES * RAW_BYTES +
                                E_RING + C_RING + N_BARS * 8 + T * HEADS * 4 + 64;
    static_assert(!KFP4 || (FP8 && T == 1), "FP4 keys: E4M3 queries, decode groups");
};
}  // namespace idx

// Score of one (key, token): the head sum sum_h sq[h] * acc[h] over the 64
// accumulator columns (lo = heads 0-31, hi = heads 32-63) with paired FMAs,
// times the key scale; stored if key < nv (the token's visible entries; -1
// for a token past the end of the rows) as fp32, or rounded to bf16 (nearest
// even) when sbf16.  RELU clips each head's accumulator at 0 first (sq[h]
// then also carries the head's weight).  Returns the stored value.
template <bool RELU>
__device__ __forceinline__ float idx_store_score(uint32_t (&lo)[32], uint32_t (&hi)[32],
                                                 const float* __restrict__ sq, float sk, int key, int nv,
                                                 void* __restrict__ srow_ptr, bool sbf16)
{
    if constexpr (RELU) {
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            lo[h] = __float_as_uint(fmaxf(__uint_as_float(lo[h]), 0.f));
            hi[h] = __float_as_uint(fmaxf(__uint_as_float(hi[h]), 0.f));
        }
    }
    const float4* sq4 = reinterpret_cast<const float4*>(sq);
    uint64_t pa = 0, pb = 0, pc = 0, pd = 0;   // packed partial sums (x, y halves)
#pragma unroll
    for (int h4 = 0; h4 < 8; ++h4) {
        const float4 w4 = sq4[h4];
        const float4 u4 = sq4[8 + h4];
        pa = ffma2(pack_f32x2(w4.x, w4.y), pack_u32x2(lo[4 * h4], lo[4 * h4 + 1]), pa);
        pb = ffma2(pack_f32x2(w4.z, w4.w), pack_u32x2(lo[4 * h4 + 2], lo[4 * h4 + 3]), pb);
        pc = ffma2(pack_f32x2(u4.x, u4.y), pack_u32x2(hi[4 * h4], hi[4 * h4 + 1]), pc);
        pd = ffma2(pack_f32x2(u4.z, u4.w), pack_u32x2(hi[4 * h4 + 2], hi[4 * h4 + 3]), pd);
    }
    const float2 fa = unpack_f32x2(pa), fb = unpack_f32x2(pb), fc = unpack_f32x2(pc), fd = unpack_f32x2(pd);
    float sc = (((fa.x + fa.y) + (fb.x + fb.y)) + ((fc.x + fc.y) + (fd.x + fd.y))) * sk;
    if (sbf16) {
        const __nv_bfloat16 h = __float2bfloat16_rn(sc);
        if (key < nv) reinterpret_cast<__nv_bfloat16*>(srow_ptr)[key] = h;
        sc = __bfloat162float(h);
    } else if (key < nv) {
        reinterpret_cast<float*>(srow_ptr)[key] = sc;
    }
    return sc;
}

// Row scale of an FP4 key from its four E4M3 block scales (one word, block 0
// in the low byte): S = 2^(floor(log2 max_b sc_b) - 5), and 1 / S.
__device__ __forceinline__ void fp4_row_scale(uint32_t sw, float& S, float& inv_S)
{
    const float2 a = e4m3x2_to_f32x2((uint16_t)(sw & 0xFFFFu)), c = e4m3x2_to_f32x2((uint16_t)(sw >> 16));
    const float mx = fmaxf(fmaxf(fmaxf(0.f, a.x), a.y), fmaxf(c.x, c.y));
    const int ex = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;   // floor(log2 mx), mx normal
    S = __uint_as_float((uint32_t)(127 + (ex - 5)) << 23);
    inv_S = __uint_as_float((uint32_t)(127 - (ex - 5)) << 23);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Eight E2M1 codes (nibble i = element i) -> eight E4M3 bytes (byte i of
// out[0..1] = element i) through the block's magnitude table (tab_lo: bytes
// for |e| = 0, 0.5, 1, 1.5; tab_hi: 2, 3, 4, 6).  A selector nibble with its
// top bit set makes the permute return 0xFF (the sign of 0x80 replicated),
// else 0x80; shifted left by one, bit 7 of each byte then holds the code's
// sign, which flips the looked-up byte's.
__device__ __forceinline__ void e2m1x8_to_e4m3x8(uint32_t w, uint32_t tab_lo, uint32_t tab_hi, uint32_t& o0,
                                                 uint32_t& o1)
{
    const uint32_t w1 = w >> 16;
    const uint32_t p0 = prmt(tab_lo, tab_hi, w & 0x7777u), m0 = prmt(0x80808080u, 0x80808080u, w);
    const uint32_t p1 = prmt(tab_lo, tab_hi, w1 & 0x7777u), m1 = prmt(0x80808080u, 0x80808080u, w1);
    o0 = p0 ^ ((m0 << 1) & 0x80808080u);
    o1 = p1 ^ ((m1 << 1) & 0x80808080u);
}

// One 32-element block of an FP4 key (16 packed bytes, block scale sc, the
// row's 1 / S) -> 32 E4M3 bytes, E4M3(e * sc / S) each.  e * sc / S is exact
// in fp32 (a 2-bit by 4-bit significand product times a power of two), so
// the table entry equals the per-element conversion.
__device__ __forceinline__ void fp4_block_to_e4m3(const uint4& v, float sc, float inv_S, uint32_t (&o)[8])
{
    const float r = __fmul_rn(sc, inv_S);
    const uint32_t t01 = f32x2_to_e4m3x2(__fmul_rn(0.f, r), __fmul_rn(0.5f, r));
    const uint32_t t23 = f32x2_to_e4m3x2(r, __fmul_rn(1.5f, r));
    const uint32_t t45 = f32x2_to_e4m3x2(__fmul_rn(2.f, r), __fmul_rn(3.f, r));
    const uint32_t t67 = f32x2_to_e4m3x2(__fmul_rn(4.f, r), __fmul_rn(6.f, r));
    const uint32_t tab_lo = t01 | (t23 << 16), tab_hi = t45 | (t67 << 16);
    e2m1x8_to_e4m3x8(v.x, tab_lo, tab_hi, o[0], o[1]);
    e2m1x8_to_e4m3x8(v.y, tab_lo, tab_hi, o[2], o[3]);
    e2m1x8_to_e4m3x8(v.z, tab_lo, tab_hi, o[4], o[5]);
    e2m1x8_to_e4m3x8(v.w, tab_lo, tab_hi, o[6], o[7]);
}

// WMAX (decode groups, T = 1): for every 32 consecutive keys of a row (one
// epilogue warp's share of a tile) the largest score key (score_key) is also
// written to wmax[row * wmax_ld + key / 32].  The k-th largest of a row's warp
// maxima bounds its k-th largest score from below with at least k entries at
// or above it, so the top-k needs no sampled threshold.  (Counting the maxima
// into a per-row histogram with global atomics instead cost the kernel about
// a quarter of its time: the hot bins serialise.)
template <bool FP8, int T, bool WMAX, bool KFP4>
__global__ void __launch_bounds__(idx::threads<T, KFP4>(), KFP4 ? 2 : 1) indexer_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const float* __restrict__ q_scale, const float* __restrict__ head_w, int relu, const float* __restrict__ k_scale,
    void* __restrict__ scores, int score_bf16, int n_q_total, int i_start, int n_q_rows, QPos qp, int m,
    int Nc, int n_splits, int split_tiles, uint32_t* __restrict__ wmax, int wmax_ld,
    uint32_t* __restrict__ zero_words, int n_zero)
{
    grid_dep_entry();
    // words the next kernel expects cleared (the top-k's row counters)
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int x = threadIdx.x; x < n_zero; x += blockDim.x) zero_words[x] = 0u;
    using C = idx::Cfg<FP8, T, KFP4>;
    static_assert(!WMAX || T == 1, "warp maxima: decode groups");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base;
    uint8_t* sK = sQ + C::Q_BYTES;
    uint8_t* sRaw = sK + C::STAGES * C::K_BYTES;            // packed FP4 tiles (KFP4)
    uint32_t* e_ring = reinterpret_cast<uint32_t*>(sRaw + C::RAW_STAGES * C::RAW_BYTES);
    uint32_t* c_ring = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(e_ring) + C::E_RING);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(c_ring) + C::C_RING);
    uint64_t* bar_full = bars;
    uint64_t* bar_empty = bars + C::STAGES;
    uint64_t* bar_acc_full = bars + 2 * C::STAGES;
    uint64_t* bar_acc_empty = bars + 2 * C::STAGES + C::ACC;
    uint64_t* bar_q = bars + 2 * C::STAGES + 2 * C::ACC;
    uint64_t* bar_mma_done = bar_q + 1;
    uint64_t* bar_raw_full = bar_mma_done + 1;
    uint64_t* bar_raw_empty = bar_raw_full + C::RAW_STAGES;
    float* sq_s = reinterpret_cast<float*>(bars + C::N_BARS);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sq_s + T * idx::HEADS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int g = blockIdx.x / n_splits, split = blockIdx.x % n_splits;
    const int i0 = g * T;                                   // first token of the group (chunk-local)
    const int i_last = min(i0 + T - 1, n_q_rows - 1);
    const long long q_pos0 = qp.at(blockIdx.y);   // this sequence's first query position
    long long nvl = (q_pos0 + i_start + i_last + 1) / m;
    const int nv_last = (int)(nvl < Nc ? nvl : Nc);
    const int total_tiles = (nv_last + idx::BLOCK_KEYS - 1) / idx::BLOCK_KEYS;
    const int tile0 = split * split_tiles;
    const int n_tiles = min(split_tiles, total_tiles - tile0);
    if (n_tiles <= 0) return;  // uniform over the CTA

    if (threadIdx.x == 0) {
        // KFP4: the converter warps, not the copy engine, fill the operand stages
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&bar_full[s], KFP4 ? idx::CONV_WARPS : 1);
            mbar_init(&bar_empty[s], 1);
        }
        for (int s = 0; s < C::RAW_STAGES; ++s) {
            mbar_init(&bar_raw_full[s], 1);
            mbar_init(&bar_raw_empty[s], idx::CONV_WARPS);
        }
        for (int a = 0; a < C::ACC; ++a) {
            mbar_init(&bar_acc_full[a], 1);
            mbar_init(&bar_acc_empty[a], idx::epi_warps<T>());
        }
        mbar_init(bar_q, 1);
        mbar_init(bar_mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            const int qrow = (b * n_q_total + i_start + i0) * idx::HEADS;
            mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
            for (int a = 0; a < C::ATOMS; ++a)
                tma_load_2d(sQ + a * C::Q_ATOM, &tmap_q, bar_q, a * (idx::ATOM_BYTES_ROW / C::ELEM), qrow);
            int issued = 0;
            // decode groups read each key tile once: mark its lines first for
            // eviction, so the stream leaves the scores (which the top-k reads
            // next) in L2
            const uint64_t kpol = l2_policy_evict_first();
            if constexpr (KFP4) {
                // packed tiles into the raw ring; the converter warps free its stages
                for (int li = 0; li < n_tiles; ++li) {
                    const int rs = li % C::RAW_STAGES;
                    if (!mbar_wait(&bar_raw_empty[rs], ((li / C::RAW_STAGES) & 1) ^ 1, abort_flag)) break;
                    mbar_arrive_expect_tx(&bar_raw_full[rs], C::RAW_BYTES);
                    tma_load_2d_hint(sRaw + rs * C::RAW_BYTES, &tmap_k, &bar_raw_full[rs], 0,
                                     b * Nc + (tile0 + li) * idx::BLOCK_KEYS, kpol);
                    issued = li + 1;
                }
            } else {
                for (int li = 0; li < n_tiles; ++li) {
                    const int st = li % C::STAGES;
                    const uint32_t ph = (li / C::STAGES) & 1;
                    if (!mbar_wait(&bar_empty[st], ph ^ 1, abort_flag)) break;
                    mbar_arrive_expect_tx(&bar_full[st], C::K_BYTES);
                    const int krow = b * Nc + (tile0 + li) * idx::BLOCK_KEYS;
                    uint8_t* dst = sK + st * C::K_BYTES;
                    for (int a = 0; a < C::ATOMS; ++a) {
                        if constexpr (T == 1)
                            tma_load_2d_hint(dst + a * C::K_ATOM, &tmap_k, &bar_full[st],
                                             a * (idx::ATOM_BYTES_ROW / C::ELEM), krow, kpol);
                        else
                            tma_load_2d(dst + a * C::K_ATOM, &tmap_k, &bar_full[st], a * (idx::ATOM_BYTES_ROW / C::ELEM), krow);
                    }
                    issued = li + 1;
                }
            }
            if (*abort_flag) {
                // let copies already in flight land before the CTA exits
                mbar_wait(bar_q, 0);
                if constexpr (KFP4) {
                    for (int li = max(0, issued - C::RAW_STAGES); li < issued; ++li)
                        mbar_wait(&bar_raw_full[li % C::RAW_STAGES], (li / C::RAW_STAGES) & 1);
                } else {
                    for (int li = max(0, issued - C::STAGES); li < issued; ++li)
                        mbar_wait(&bar_full[li % C::STAGES], (li / C::STAGES) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (one thread) ----------------
        if (lane == 0) {
            const uint32_t sQ_addr = smem_u32(sQ);
            const uint32_t sK_addr = smem_u32(sK);
            if (mbar_wait(bar_q, 0, abort_flag)) {
                for (int li = 0; li < n_tiles; ++li) {
                    const int st = li % C::STAGES;
                    const int acc = li % C::ACC;
                    if (!mbar_wait(&bar_full[st], (li / C::STAGES) & 1, abort_flag)) break;
                    if (!mbar_wait(&bar_acc_empty[acc], ((li / C::ACC) & 1) ^ 1, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * C::N;
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS; ++ks) {
                        const int atom = ks / C::KSTEPS_PER_ATOM;
                        const uint32_t koff = (ks % C::KSTEPS_PER_ATOM) * 32;
                        const uint64_t a_desc = smem_desc(sK_addr + st * C::K_BYTES + atom * C::K_ATOM + koff, 16, 1024, SWZ_128B);
                        const uint64_t b_desc = smem_desc(sQ_addr + atom * C::Q_ATOM + koff, 16, 1024, SWZ_128B);
                        if constexpr (FP8) umma_f8(d_tmem, a_desc, b_desc, C::IDESC, ks > 0);
                        else umma_f16(d_tmem, a_desc, b_desc, C::IDESC, ks > 0);
                    }
                    umma_commit(&bar_empty[st]);
                    umma_commit(&bar_acc_full[acc]);
                }
            }
            umma_commit(bar_mma_done);       // all MMAs of this CTA retired
            mbar_wait(bar_mma_done, 0);
        }
    } else if (warp >= 2 + idx::epi_warps<T>()) {
        // ---------------- FP4 -> E4M3 converters (KFP4 only) ----------------
        if constexpr (KFP4) {
        // Thread ct takes items ct + 128 r (r < 4) of a tile, item = 4 * key +
        // block: a warp reads 512 contiguous packed bytes and writes each
        // item's 32 E4M3 bytes as two 16-byte chunks of the key's 128-byte
        // row, XOR-swizzled by key % 8 (the 128-byte swizzle of the operand).
        // The keys' scale words come SC_DEPTH - 1 tiles ahead by cp.async.
        constexpr int NCT = 32 * idx::CONV_WARPS, NI = idx::CONV_ITEMS;
        static_assert(NI == 4, "one 16-byte ring read a thread a tile");
        const int ct = threadIdx.x - 32 * (2 + idx::epi_warps<T>());
        const int blk = ct & 3;
        const uint32_t* scw = reinterpret_cast<const uint32_t*>(k_scale) + (long long)b * Nc;
        auto c_issue = [&](int lj) {
            uint32_t* dst = c_ring + ((lj % idx::SC_DEPTH) * NCT + ct) * NI;
#pragma unroll
            for (int r = 0; r < NI; ++r) {
                const int key = (tile0 + lj) * idx::BLOCK_KEYS + ((ct + NCT * r) >> 2);
                if (lj < n_tiles && key < Nc) cp_async4(dst + r, scw + key);
                else dst[r] = 0x38383838u;                  // E4M3 1.0 past the end
            }
            cp_async_commit();
        };
        for (int lj = 0; lj < idx::SC_DEPTH - 1; ++lj) c_issue(lj);
        for (int li = 0; li < n_tiles; ++li) {
            c_issue(li + idx::SC_DEPTH - 1);
            const int rs = li % C::RAW_STAGES;
            const bool ok = mbar_wait(&bar_raw_full[rs], (li / C::RAW_STAGES) & 1, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            uint4 v[NI];
#pragma unroll
            for (int r = 0; r < NI; ++r)
                v[r] = *reinterpret_cast<const uint4*>(sRaw + rs * C::RAW_BYTES + (ct + NCT * r) * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_raw_empty[rs]);
            cp_async_wait<idx::SC_DEPTH - 1>();
            const uint4 sw4 = *reinterpret_cast<const uint4*>(c_ring + ((li % idx::SC_DEPTH) * NCT + ct) * NI);
            const uint32_t sw[NI] = {sw4.x, sw4.y, sw4.z, sw4.w};
            const int st = li % C::STAGES;
            const bool ok2 = mbar_wait(&bar_empty[st], ((li / C::STAGES) & 1) ^ 1, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, ok2)) break;
#pragma unroll
            for (int r = 0; r < NI; ++r) {
                float S, inv_S;
                fp4_row_scale(sw[r], S, inv_S);
                const float scb = e4m3x2_to_f32x2((uint16_t)((sw[r] >> (8 * blk)) & 0xFFu)).x;
                uint32_t o[8];
                fp4_block_to_e4m3(v[r], scb, inv_S, o);
                const int key = (ct + NCT * r) >> 2;
                uint8_t* row = sK + st * C::K_BYTES + key * idx::ATOM_BYTES_ROW;
                *reinterpret_cast<uint4*>(row + (((2 * blk) ^ (key & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(row + (((2 * blk + 1) ^ (key & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_smem();   // generic-proxy writes, read next by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_full[st]);
        }
        cp_async_wait<0>();             // no copy outlives the loop
        }
    } else {
        // ---------------- epilogue: one TMEM lane (= key) per thread ----------------
        // Warp w (w >= 2) reads lane quadrant w % 4 and takes token (w - 2) / 4
        // of the group.  Both halves of its 64 columns are loaded before one
        // wait; the head sum uses paired FMAs in four independent chains.
        constexpr int EW = idx::epi_warps<T>();
        const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const int ew = warp - 2;                   // 0..EW-1
        const int tt0 = ew / 4;                    // this warp's token within the group
        const int et = threadIdx.x - 64;           // 0..32*EW-1
        for (int x = et; x < T * idx::HEADS; x += 32 * EW) {
            const int tt = x / idx::HEADS, h = x % idx::HEADS;
            const int i = i0 + tt;
            float v = 0.f;
            if (i < n_q_rows) {
                const long long qh = ((long long)b * n_q_total + i_start + i) * idx::HEADS + h;
                v = q_scale ? q_scale[qh] : 1.f;
                if (head_w) v *= head_w[qh];   // weighted variant: the head's weight joins its scale
            }
            sq_s[x] = v;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
        // this warp's token: visible entries (constant over the tiles) and score row
        const int i_tok = i0 + tt0;
        int nv_tok = -1;
        if (i_tok < n_q_rows) {
            const long long nvl_t = (q_pos0 + i_start + i_tok + 1) / m;
            nv_tok = (int)(nvl_t < Nc ? nvl_t : Nc);
        }
        const bool sbf16 = score_bf16 != 0;
        void* const srow_ptr = reinterpret_cast<uint8_t*>(scores) +
                               ((long long)b * n_q_rows + (i_tok < n_q_rows ? i_tok : 0)) * Nc * (sbf16 ? 2 : 4);
        // key scales: fp32 row scales, or (KFP4) the words of four E4M3 block
        // scales; decode groups copy them SC_DEPTH - 1 tiles ahead by cp.async
        const uint32_t* ksw = k_scale ? reinterpret_cast<const uint32_t*>(k_scale) + (long long)b * Nc : nullptr;
        constexpr uint32_t ONE = KFP4 ? 0x38383838u : 0x3F800000u;
        auto e_issue = [&](int lj) {
            uint32_t* dst = e_ring + (lj % idx::SC_DEPTH) * (32 * EW) + et;
            const int kj = (tile0 + lj) * idx::BLOCK_KEYS + row;
            if (k_scale && lj < n_tiles && kj < Nc) cp_async4(dst, ksw + kj);
            else *dst = ONE;
            cp_async_commit();
        };
        if constexpr (C::SC_RING)
            for (int lj = 0; lj < idx::SC_DEPTH - 1; ++lj) e_issue(lj);
        for (int li = 0; li < n_tiles; ++li) {
            const int acc = li % C::ACC;
            const int key = (tile0 + li) * idx::BLOCK_KEYS + row;
            uint32_t sw;
            if constexpr (C::SC_RING) {
                e_issue(li + idx::SC_DEPTH - 1);
                cp_async_wait<idx::SC_DEPTH - 1>();
                sw = e_ring[(li % idx::SC_DEPTH) * (32 * EW) + et];
            } else {
                sw = (k_scale && key < Nc) ? __ldg(ksw + key) : ONE;
            }
            float sk;
            if constexpr (KFP4) {   // the row scale S, from the key's block scales
                float inv_S;
                fp4_row_scale(sw, sk, inv_S);
            } else {
                sk = __uint_as_float(sw);
            }
            const bool ok = mbar_wait(&bar_acc_full[acc], (li / C::ACC) & 1, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;   // tcgen05.ld below is warp-collective
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * C::N + tt0 * idx::HEADS;
            uint32_t va[32], vb[32];   // heads 0-31 | 32-63 of this warp's token
            tmem_ld32(tbase, va);
            tmem_ld32(tbase + 32, vb);
            tmem_ld_wait();
            // the accumulator can be refilled once the registers hold it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_acc_empty[acc]);
            const float sc = relu ? idx_store_score<true>(va, vb, sq_s + tt0 * idx::HEADS, sk, key, nv_tok, srow_ptr, sbf16)
                                  : idx_store_score<false>(va, vb, sq_s + tt0 * idx::HEADS, sk, key, nv_tok, srow_ptr, sbf16);
            if constexpr (WMAX) {
                const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, key < nv_tok ? score_key(sc) : 0u);
                const int grp = (tile0 + li) * (idx::BLOCK_KEYS / 32) + quad;   // keys 32 grp .. 32 grp + 31
                if (lane == 0 && grp * 32 < nv_tok) wmax[((long long)b * n_q_rows + i_tok) * wmax_ld + grp] = mx;
            }
        }
        if constexpr (C::SC_RING) cp_async_wait<0>();   // no copy outlives the loop
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// fp32 scores on CUDA cores (any H_I, d_I): one thread per (query, entry).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) indexer_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ q_scale, const float* __restrict__ head_w, int relu,
    const float* __restrict__ k, const float* __restrict__ k_scale, void* __restrict__ scores, int score_bf16,
    int n_q_total, int i_start, int n_q_rows, QPos qp, int m, int Nc, int HI, int dI)
{
    grid_dep_entry();
    extern __shared__ float qs[];
    const int r = blockIdx.y;          // chunk-local row = b * n_q_rows + i
    const int b = r / n_q_rows, i = r % n_q_rows;
    const long long qrow = (long long)b * n_q_total + i_start + i;
    for (int x = threadIdx.x; x < HI * dI; x += blockDim.x) qs[x] = q[qrow * HI * dI + x];
    for (int x = threadIdx.x; x < HI; x += blockDim.x)
        qs[HI * dI + x] = (q_scale ? q_scale[qrow * HI + x] : 1.f) * (head_w ? head_w[qrow * HI + x] : 1.f);
    __syncthreads();
    long long nvl = (qp.at(b) + i_start + i + 1) / m;
    const int nv = (int)(nvl < Nc ? nvl : Nc);
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= nv) return;
    const float* kr = k + ((long long)b * Nc + j) * dI;
    const float sk = k_scale ? k_scale[(long long)b * Nc + j] : 1.f;
    float s = 0.f;
    for (int h = 0; h < HI; ++h) {
        float dot = 0.f;
        for (int c = 0; c < dI; ++c) dot = fmaf(qs[h * dI + c], __ldg(kr + c), dot);
        if (relu) dot = fmaxf(dot, 0.f);
        s = fmaf(qs[HI * dI + h] * sk, dot, s);
    }
    if (score_bf16) reinterpret_cast<__nv_bfloat16*>(scores)[(long long)r * Nc + j] = __float2bfloat16_rn(s);
    else reinterpret_cast<float*>(scores)[(long long)r * Nc + j] = s;
}

// ---------------------------------------------------------------------------
// FP4 (E2M1) -> FP8 (E4M3) widening of indexer keys ("DeepSeek V4 技术解读"
// §五): per row S = 2^(floor(log2 max_b sc_b) - 5); x8 = E4M3(e * sc_b / S).
// e * sc_b is exact in fp32 and S is a power of two, so the E4M3 conversion
// is the only rounding.  One thread per 32-element block.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fp4_to_e4m3_kernel(const uint8_t* __restrict__ packed,
                                                          const uint8_t* __restrict__ sc,
                                                          uint8_t* __restrict__ x8, float* __restrict__ S,
                                                          long long rows, int d)
{
    grid_dep_entry();
    const int nb = d / 32;
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * nb) return;
    const long long r = t / nb;
    const int blk = (int)(t % nb);
    float mx = 0.f;
    for (int q = 0; q < nb; ++q) mx = fmaxf(mx, e4m3x2_to_f32x2(sc[r * nb + q]).x);
    const int ex = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;   // floor(log2 mx), mx normal
    const float inv_S = __uint_as_float((uint32_t)(127 - (ex - 5)) << 23);
    const float scb = e4m3x2_to_f32x2(sc[r * nb + blk]).x;
    const uint4 p = *reinterpret_cast<const uint4*>(packed + r * (d / 2) + blk * 16);
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
    uint32_t outw[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float v[8];
        e2m1x8_to_f32x8(w[q], v);
#pragma unroll
        for (int c = 0; c < 8; c += 4) {
            const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(__fmul_rn(v[c], scb), inv_S),
                                                __fmul_rn(__fmul_rn(v[c + 1], scb), inv_S));
            const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(__fmul_rn(v[c + 2], scb), inv_S),
                                                __fmul_rn(__fmul_rn(v[c + 3], scb), inv_S));
            outw[2 * q + c / 4] = lo | (hi << 16);
        }
    }
    uint4* o = reinterpret_cast<uint4*>(x8 + r * d + blk * 32);
    o[0] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
    o[1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    if (blk == 0) S[r] = __uint_as_float((uint32_t)(127 + (ex - 5)) << 23);
}

cudaError_t launch_fp4_to_e4m3(const uint8_t* packed, const uint8_t* sc, uint8_t* x8, float* S,
                               long long rows, int d, cudaStream_t s)
{
    const long long n = rows * (d / 32);
    if (n == 0) return cudaSuccess;
    (void)launch_pdl(fp4_to_e4m3_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, packed, sc, x8, S, rows, d);
    return cudaGetLastError();
}

cudaError_t launch_indexer_f32(const float* q, const float* q_scale, const float* head_w, bool relu,
                               const float* k, const float* k_scale, void* scores, bool score_bf16, int B,
                               int n_q_total, int i_start, int n_q_rows, QPos q_pos0, int m, int Nc, int HI,
                               int dI, cudaStream_t s)
{
    if (B * n_q_rows == 0 || Nc == 0) return cudaSuccess;
    dim3 grid((Nc + 255) / 256, B * n_q_rows);
    size_t smem = (size_t)(HI * dI + HI) * sizeof(float);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(indexer_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    (void)launch_pdl(indexer_f32_kernel, dim3(grid), dim3(256), smem, s, q, q_scale, head_w, relu ? 1 : 0, k, k_scale, scores, score_bf16 ? 1 : 0, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, HI, dI);
    return cudaGetLastError();
}

template <bool FP8, int T, bool WMAX, bool KFP4 = false>
static cudaError_t launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const float* q_scale, const float* head_w,
                             bool relu, const float* k_scale, void* scores, bool score_bf16, int B, int n_q_total,
                             int i_start,
                             int n_q_rows, QPos q_pos0, int m, int Nc, int num_sms, uint32_t* wmax,
                             int wmax_ld, cudaStream_t s, uint32_t* zero_words = nullptr, int n_zero = 0)
{
    using C = idx::Cfg<FP8, T, KFP4>;
    const int n_groups = (n_q_rows + T - 1) / T;
    // per-sequence positions live on the device: cover every entry
    long long nv_max = q_pos0.lens ? (long long)Nc : (q_pos0.q_pos0 + i_start + n_q_rows) / m;
    if (nv_max > Nc) nv_max = Nc;
    const int tiles = (int)((nv_max + idx::BLOCK_KEYS - 1) / idx::BLOCK_KEYS);
    if (tiles == 0 || n_groups == 0) return cudaSuccess;
    // split the key range when there are too few query groups to fill the GPU
    const int per_sm = (C::SMEM <= 113 * 1024) ? 2 : 1;
    // waves of CTAs: 12 for E4M3 keys (a sweep of 3-16 at batch 32: 12 best,
    // 0.2015 -> 0.1935 ms for index + top-k), 4 for the widening E2M1 route
    // (12 there: 0.278 -> 0.296 ms)
    // (12 waves only while a CTA keeps at least 16 key tiles: small batches
    // would otherwise spend more on per-CTA set-up than they gain)
    const long long target = (long long)num_sms * per_sm * (KFP4 ? 4 : 12);
    int splits = (int)std::min<long long>(tiles, std::max<long long>(1, (target + (long long)B * n_groups - 1) / ((long long)B * n_groups)));
    if (!KFP4) splits = std::max(1, std::min(splits, tiles / 16));
    const int split_tiles = (tiles + splits - 1) / splits;
    splits = (tiles + split_tiles - 1) / split_tiles;
    auto kern = indexer_tc_kernel<FP8, T, WMAX, KFP4>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    dim3 grid(n_groups * splits, B);
    (void)launch_pdl(kern, dim3(grid), dim3(idx::threads<T, KFP4>()), C::SMEM, s, tq, tk, q_scale, head_w, relu ? 1 : 0, k_scale, scores, score_bf16 ? 1 : 0, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, splits, split_tiles, wmax, wmax_ld, zero_words, n_zero);
    return cudaGetLastError();
}

cudaError_t launch_indexer_tc(bool fp8, int T, const CUtensorMap& tq, const CUtensorMap& tk,
                              const float* q_scale, const float* head_w, bool relu, const float* k_scale,
                              void* scores, bool score_bf16, int B,
                              int n_q_total, int i_start, int n_q_rows, QPos q_pos0, int m, int Nc,
                              int num_sms, uint32_t* wmax, int wmax_ld, bool kfp4, cudaStream_t s,
                              uint32_t* zero_words, int n_zero)
{
    if (kfp4) {   // packed E2M1 keys widened in the kernel: E4M3 queries, decode groups
        if (!fp8 || T != 1) return cudaErrorInvalidValue;
        if (wmax) return launch_tc<true, 1, true, true>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, wmax, wmax_ld, s, zero_words, n_zero);
        return launch_tc<true, 1, false, true>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, nullptr, 0, s);
    }
    if (wmax) {   // decode groups (T = 1) only
        if (T != 1) return cudaErrorInvalidValue;
        if (fp8) return launch_tc<true, 1, true>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, wmax, wmax_ld, s, zero_words, n_zero);
        return launch_tc<false, 1, true>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, wmax, wmax_ld, s, zero_words, n_zero);
    }
    if (fp8) {
        if (T == 4) return launch_tc<true, 4, false>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, nullptr, 0, s);
        return launch_tc<true, 1, false>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, nullptr, 0, s);
    }
    if (T == 4) return launch_tc<false, 4, false>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, nullptr, 0, s);
    return launch_tc<false, 1, false>(tq, tk, q_scale, head_w, relu, k_scale, scores, score_bf16, B, n_q_total, i_start, n_q_rows, q_pos0, m, Nc, num_sms, nullptr, 0, s);
}

int indexer_group_tokens(int n_q) { return n_q >= 4 ? 4 : 1; }
int indexer_box_rows(int T) { return idx::HEADS * T; }

}  // namespace csa
