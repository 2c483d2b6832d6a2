// Attention of H query heads over one shared KV head on the tcgen05 tensor
// cores (BF16 in, fp32 accumulate), for the three key sets of the hybrid
// stack ("DeepSeek V4 技术解读"):
//   mode 0  CSA core attention over the top-k selected entries (§2.1 Core
//           Attention), the selected entries fetched with TMA row gathers,
//   mode 1  HCA dense attention over all closed compressed blocks (§2.2),
//   mode 2  sliding-window attention over raw tokens (§2.3).
//
// One CTA owns 128 (token, head) rows -- the M side of both products -- and
// walks its key set in tiles of 128 keys:
//     S   = Q K^T   A = Q  [128 rows x 128 dims]  smem, K-major, 128B swizzle
//                   B = K  [128 keys x 128 dims]  smem, K-major
//                   D = S  [128 lanes x 128 cols] fp32 in tensor memory
//     O  += P V     A = P  [128 rows x 128 keys]  bf16 in tensor memory, over S
//                   B = V  [128 keys x 128 dims]  smem, read MN-major
//                   D = O  [128 lanes x 128 cols] fp32 in tensor memory
// With every head in the M dimension each TMEM lane is one (token, head) row,
// so the softmax (max, exponentials, row sum) is a per-thread loop with no
// cross-thread reduction.  Rows are 2 tokens x 64 heads (dense modes) or one
// token x H heads (sparse mode: every token has its own key set; with H = 64
// the upper 64 rows idle).
//
// Warp roles.  Dense modes (224 threads):
//   warps 0-1  producer: Q once, then K and V tiles into rings of STAGES
//              buffers by tiled TMA (a K stage is released when S_j
//              completes, a V stage when P_j V_j completes);
//   warp 2     TMEM owner and single-thread MMA issuer: S_j into one of two S
//              buffers, then O += P_{j-1} V_{j-1}, so the QK^T of tile j
//              overlaps the softmax of tile j-1;
//   warps 3-6  softmax and epilogue, one row per thread: online softmax in
//              the base-2 domain against a lazily moved reference maximum,
//              P written back to TMEM as bf16; O and l are rescaled (in TMEM)
//              only when a row's maximum grows by more than 2^8.
// Sparse mode (512 threads): the selected rows are scattered, and fetching
// them sets the pace, so eleven warps gather them with 16-byte cp.async
// (about 1.8x the rate of TMA tile::gather4 from two warps on an L2-resident
// table: 23.7 vs 12.9 bytes per cycle per SM, measured on B300); each gather
// warp publishes tile j after issuing tile j+1, once its own copies of tile j
// have landed (cp.async.wait_group, then a proxy fence, then its arrival) --
// or at once, before blocking on the ring, when no stage is free for tile j+1.
//   warps 0-3  softmax and epilogue, two passes over 32-column chunks of S
//              (row maximum, then exponentials) so that they fit the 128
//              registers a thread of a 512-thread CTA has;
//   warp 4     TMEM owner and MMA issuer, as above;
//   warps 5-15 gather warps: Q by TMA once, the CTA's selection list into
//              shared memory, then the K and V rows of every tile (eleven
//              warps instead of eight: 32K prefill 4.10 -> 3.99 ms).
// Every mbarrier wait is bounded; on a timeout the CTA drains its copies and
// MMAs, frees TMEM and exits with the device status word set.
//
// Split key sets (decode-shaped calls) write unnormalised partials (o, m, l)
// that attn_combine_kernel merges in split order, so results stay
// deterministic and independent of the batch size.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace atc {
// warp roles per mode (see the header)
template <int MODE> struct Roles {
    static constexpr bool SPARSE = MODE == 0;
    static constexpr int THREADS = SPARSE ? 512 : 224;
    static constexpr int MMA_WARP = SPARSE ? 4 : 2;
    static constexpr int SOFTMAX_WARP0 = SPARSE ? 0 : 3;   // four consecutive warps
    static constexpr int GATHER_WARP0 = 5;                  // sparse mode: every warp after the MMA warp
    static constexpr int GATHER_WARPS = 11;
};
static_assert(Roles<0>::GATHER_WARP0 + Roles<0>::GATHER_WARPS <= Roles<0>::THREADS / 32 &&
                  Roles<0>::GATHER_WARP0 > Roles<0>::MMA_WARP, "gather warps inside the CTA, after the others");
constexpr int ROWS = 128;                 // MMA M
constexpr int KT = 128;                   // keys per tile
constexpr int D = 128;                    // head dim
constexpr int ATOM = 128 * 128;           // 128 rows x 128 bytes (64 bf16 columns)
constexpr int K_BYTES = 2 * ATOM;
constexpr int V_BYTES = 2 * ATOM;
constexpr int S_COL = 0;                  // S buffers at columns 0 (and 128)
// SBUFS S buffers (1 or 2), then the O accumulator; the allocation is the
// next power of two (two S buffers: 512 columns, one CTA an SM; one S
// buffer: 256 columns, so two CTAs share an SM's tensor memory)
constexpr int o_col(int sbufs) { return sbufs * KT; }
constexpr int tmem_cols(int sbufs) { return sbufs == 1 ? 256 : 512; }
constexpr uint32_t IDESC_S = instr_desc(1u, 1u, ROWS, KT);          // bf16, both K-major
constexpr uint32_t IDESC_PV = instr_desc(1u, 1u, ROWS, D, 0u, 1u);  // B (= V) MN-major
constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr int MAX_LIST = 4096;            // selected entries one CTA stages (sparse mode)
constexpr int SMALL_MAX_TILES = 8;        // dense key sets of at most this many tiles: the small configuration

// QROWS: Q rows loaded per CTA.  With 64 (one token of 64 heads) the two
// 64-column Q blocks sit 8 KB apart; the MMA still reads 128 rows, and rows
// 64..127 (which read neighbouring data) only feed unused accumulator lanes.
template <int MODE, int STAGES, int QROWS> struct Cfg {
    static constexpr int Q_ATOM = QROWS * 128;
    static constexpr int Q_BYTES = 2 * Q_ATOM;
    static constexpr int LIST = MODE == 0 ? MAX_LIST : 0;
    // barriers: q, mma_done, list, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_full[2], o_full
    static constexpr int N_BARS = 3 + 4 * STAGES + 5;
    static constexpr int SMEM = 1024 + Q_BYTES + STAGES * (K_BYTES + V_BYTES) + LIST * 4 + N_BARS * 8 + 16;
    static_assert(SMEM <= 232448, "shared memory");
};
}  // namespace atc

// SBUFS = 1 (dense modes, one ring stage): the small configuration for short
// key sets, two CTAs an SM -- S_j is issued only after P_{j-1} V_{j-1} has
// completed, and one CTA's set-up and loads overlap the other's work.
template <int MODE, int STAGES, int QROWS, int SBUFS>
__global__ void __launch_bounds__(atc::Roles<MODE>::THREADS, SBUFS == 1 ? 2 : 1) attn_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
    const __grid_constant__ CUtensorMap tmap_v, const AttnTcParams p)
{
    grid_dep_entry();
    using namespace atc;
    using C = Cfg<MODE, STAGES, QROWS>;
    using R = Roles<MODE>;
    static_assert(SBUFS == 2 || (SBUFS == 1 && !R::SPARSE), "one S buffer: dense modes");
    constexpr int O_COL = o_col(SBUFS);
    constexpr int TMEM_COLS = tmem_cols(SBUFS);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = base;
    uint8_t* sK = sQ + C::Q_BYTES;
    uint8_t* sV = sK + STAGES * K_BYTES;
    int32_t* sidx = reinterpret_cast<int32_t*>(sV + STAGES * V_BYTES);   // sparse mode: the CTA's list
    uint64_t* bars = reinterpret_cast<uint64_t*>(sidx + C::LIST);
    uint64_t* bar_q = bars;
    uint64_t* bar_mma_done = bars + 1;
    uint64_t* bar_list = bars + 2;        // sparse mode: the staged list is complete
    uint64_t* k_full = bars + 3;
    uint64_t* v_full = k_full + STAGES;
    uint64_t* k_empty = v_full + STAGES;  // K stage free once S_j has completed
    uint64_t* v_empty = k_empty + STAGES; // V stage free once P_j V_j has completed
    uint64_t* s_full = v_empty + STAGES;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_full = p_full + 2;        // one phase per completed P_j V_j
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int g = blockIdx.x / p.n_splits, split = blockIdx.x % p.n_splits;
    const int i0 = g * p.T;                                  // first query token of the CTA
    const int i_last = min(i0 + p.T, p.n_q) - 1;

    // Key range of this CTA, in list positions (mode 0) or key indices.
    long long set_lo = 0, set_len;
    if (MODE == 0) {
        set_len = p.k;
    } else if (MODE == 1) {
        const long long nv = (p.q_pos0 + i_last + 1) / p.m;
        set_len = nv < p.N_kv ? nv : p.N_kv;
    } else {
        long long lo = p.q_pos0 + i0 - p.window + 1;
        if (lo < 0) lo = 0;
        long long hi = p.q_pos0 + i_last;
        if (hi > p.N_kv - 1) hi = p.N_kv - 1;
        set_lo = lo;
        set_len = hi >= lo ? hi - lo + 1 : 0;
    }
    const long long r_lo = set_lo + (long long)split * p.split_len;
    long long r_hi = set_lo + (long long)(split + 1) * p.split_len;
    if (r_hi > set_lo + set_len) r_hi = set_lo + set_len;
    const int n_tiles = r_hi > r_lo ? (int)((r_hi - r_lo + KT - 1) / KT) : 0;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        mbar_init(bar_mma_done, 1);
        mbar_init(bar_list, 1);
        for (int s = 0; s < STAGES; ++s) {
            // sparse mode: one arrival per gather warp; dense: the TMA issuer
            mbar_init(&k_full[s], R::SPARSE ? R::GATHER_WARPS : 1);
            mbar_init(&v_full[s], R::SPARSE ? R::GATHER_WARPS : 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], 4);
        }
        mbar_init(o_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == R::MMA_WARP) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (R::SPARSE && warp >= R::GATHER_WARP0 && warp < R::GATHER_WARP0 + R::GATHER_WARPS) {
        // ------------------------- gather warps (sparse) -------------------------
        constexpr int GT = 32 * R::GATHER_WARPS;             // gather threads
        const int gl = (warp - R::GATHER_WARP0) * 32 + lane;  // 0 .. GT-1
        if (n_tiles > 0) {
            if (gl == 0) {
                tma_prefetch_desc(&tmap_q);
                const int qrow = (b * p.n_q + i0) * p.H;
                mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
                tma_load_2d(sQ, &tmap_q, bar_q, 0, qrow);
                tma_load_2d(sQ + C::Q_ATOM, &tmap_q, bar_q, 64, qrow);
            }
            // stage the CTA's slice of the selection list once (invalid -> -1),
            // padded with -1 to whole tiles
            const int32_t* sel = p.topk + ((long long)b * p.n_q + i0) * p.k;
            const int len = (int)(r_hi - r_lo), padded = n_tiles * KT;
            for (int base0 = 0; base0 < padded; base0 += GT * 4) {
                int v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = base0 + u * GT + gl;
                    v[u] = e < len ? __ldg(sel + r_lo + e) : -1;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = base0 + u * GT + gl;
                    if (e < padded) {
                        int idx = v[u];
                        if (idx >= p.N_kv || idx < -1) {
                            flag_status(STATUS_BOUNDS);
                            idx = -1;
                        }
                        sidx[e] = idx;
                    }
                }
            }
            asm volatile("bar.sync 2, %0;" ::"n"(GT) : "memory");
            if (gl == 0) mbar_arrive(bar_list);
            // K and V rows of tile j: 128 rows x 16 chunks of 16 bytes each,
            // written into the 128-byte-swizzled K-major layout (the chunk
            // index within a 128-byte row XORed with the row's low 3 bits);
            // invalid entries fetch row 0 (the softmax masks them)
            const long long bN = (long long)b * p.N_kv;
            auto gather = [&](const __nv_bfloat16* __restrict__ src, uint8_t* dst, int j) {
#pragma unroll
                for (int c0 = 0; c0 < KT * 16; c0 += GT) {
                    const int c = c0 + gl;
                    if (KT * 16 % GT != 0 && c >= KT * 16) break;
                    const int r = c >> 4, ch = c & 15;
                    const long long row = bN + max(sidx[j * KT + r], 0);
                    cp_async16(dst + (ch >> 3) * ATOM + r * 128 + (((ch & 7) ^ (r & 7)) << 4),
                               src + row * D + ch * 8);
                }
                cp_async_commit();
            };
            auto publish = [&](int j) {
                // this warp's copies of tile j have landed: make them visible
                // to the tensor cores, then arrive
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&k_full[j % STAGES]);
                    mbar_arrive(&v_full[j % STAGES]);
                }
            };
            bool ok = true;
            int published = 0;                 // tiles this warp has published
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % STAGES;
                const uint32_t par = ((j / STAGES) & 1) ^ 1;
                if (published < j) {
                    // tile j-1 is still unpublished: if the ring has no free
                    // stage for tile j yet, publish j-1 first rather than hold
                    // it behind the wait (the consumers free the stage)
                    int ready = 1;
                    if (lane == 0) ready = mbar_try_wait(&k_empty[st], par) && mbar_try_wait(&v_empty[st], par);
                    if (!__shfl_sync(FULL, ready, 0)) {
                        cp_async_wait<0>();
                        publish(j - 1);
                        published = j;
                    }
                }
                int w = 1;
                if (lane == 0) w = mbar_wait(&k_empty[st], par, abort_flag);
                if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
                gather(p.k_rows, sK + st * K_BYTES, j);
                if (lane == 0) w = mbar_wait(&v_empty[st], par, abort_flag);
                if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
                gather(p.v_rows, sV + st * V_BYTES, j);
                if (published < j) {
                    cp_async_wait<2>();        // tile j-1's two groups have landed
                    publish(j - 1);
                    published = j;
                }
            }
            cp_async_wait<0>();                // nothing of this warp is left in flight
            if (ok) publish(n_tiles - 1);
            if (gl == 0 && *abort_flag) mbar_wait(bar_q, 0);   // the Q copy lands before the CTA exits
        }
    } else if (!R::SPARSE && warp < 2) {
        // ------------------------ producer (dense modes) ------------------------
        if (n_tiles > 0 && warp == 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tmap_q);
                tma_prefetch_desc(&tmap_k);
                tma_prefetch_desc(&tmap_v);
                const int qrow = (b * p.n_q + i0) * p.H;
                mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
                tma_load_2d(sQ, &tmap_q, bar_q, 0, qrow);
                tma_load_2d(sQ + C::Q_ATOM, &tmap_q, bar_q, 64, qrow);
            }
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % STAGES;
                const uint32_t par = ((j / STAGES) & 1) ^ 1;
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&k_empty[st], par, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) break;
                const int krow = (int)((long long)b * p.N_kv + r_lo + (long long)j * KT);
                if (lane == 0) {
                    mbar_arrive_expect_tx(&k_full[st], K_BYTES);
                    tma_load_2d(sK + st * K_BYTES, &tmap_k, &k_full[st], 0, krow);
                    tma_load_2d(sK + st * K_BYTES + ATOM, &tmap_k, &k_full[st], 64, krow);
                    ok = mbar_wait(&v_empty[st], par, abort_flag);
                }
                if (!__shfl_sync(FULL, ok, 0)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&v_full[st], V_BYTES);
                    tma_load_2d(sV + st * V_BYTES, &tmap_v, &v_full[st], 0, krow);
                    tma_load_2d(sV + st * V_BYTES + ATOM, &tmap_v, &v_full[st], 64, krow);
                }
                issued = j + 1;
            }
            if (lane == 0 && *abort_flag) {
                // let the copies already in flight land before the CTA exits
                mbar_wait(bar_q, 0);
                for (int j = max(0, issued - STAGES); j < issued; ++j) {
                    mbar_wait(&k_full[j % STAGES], (j / STAGES) & 1);
                    mbar_wait(&v_full[j % STAGES], (j / STAGES) & 1);
                }
            }
        }
    } else if (warp == R::MMA_WARP) {
        // --------------------------- MMA issuer ---------------------------
        if (lane == 0 && n_tiles > 0) {
            const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
            auto issue_pv = [&](int i) -> bool {
                const int st = i % STAGES, sb = i % SBUFS;
                if (!mbar_wait(&v_full[st], (i / STAGES) & 1, abort_flag)) return false;
                if (!mbar_wait(&p_full[sb], (i / SBUFS) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint32_t a = tmem + S_COL + sb * KT;
#pragma unroll
                for (int ks = 0; ks < KT / 16; ++ks) {
                    // 16 keys per step: 2 groups of 8 key rows (SBO = 1024 B);
                    // the two 64-dim column blocks are one ATOM apart (LBO).
                    const uint64_t b_desc = smem_desc(sVa + st * V_BYTES + ks * 2048, ATOM, 1024, SWZ_128B);
                    umma_f16_tmem_a(tmem + O_COL, a + ks * 8, b_desc, IDESC_PV, (i > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&v_empty[st]);
                umma_commit(o_full);
                return true;
            };
            bool ok = mbar_wait(bar_q, 0, abort_flag);
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j % STAGES, sb = j % SBUFS;
                // the one S buffer holds P_{j-1}: issue P_{j-1} V_{j-1} first
                if (SBUFS == 1 && j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
                if (!mbar_wait(&k_full[st], (j / STAGES) & 1, abort_flag)) { ok = false; break; }
                // S buffer sb still holds P_{j - SBUFS} until P_{j - SBUFS} V_{j - SBUFS} has completed
                if (j >= SBUFS && !mbar_wait(o_full, (j - SBUFS) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + S_COL + sb * KT;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int atom = ks / 4;
                    const uint32_t koff = (ks % 4) * 32;
                    const uint64_t a_desc = smem_desc(sQa + atom * C::Q_ATOM + koff, 16, 1024, SWZ_128B);
                    const uint64_t b_desc = smem_desc(sKa + st * K_BYTES + atom * ATOM + koff, 16, 1024, SWZ_128B);
                    umma_f16(d, a_desc, b_desc, IDESC_S, ks > 0);
                }
                umma_commit(&s_full[sb]);
                umma_commit(&k_empty[st]);
                if (SBUFS == 2 && j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) issue_pv(n_tiles - 1);
            umma_commit(bar_mma_done);      // all MMAs of this CTA retired
            mbar_wait(bar_mma_done, 0);
        }
    } else if (warp >= R::SOFTMAX_WARP0 && warp < R::SOFTMAX_WARP0 + 4) {
        // ----------------------- softmax + epilogue -----------------------
        // Online softmax in the base-2 domain with a lazily moved reference
        // maximum m_ref: P_j = 2^(s * scale * log2 e - m_ref) is accumulated
        // by the tensor cores into O in TMEM; only when a row's tile maximum
        // exceeds m_ref by more than 2^8 are O and l rescaled to the new
        // maximum (so every P stays <= 256, exact enough in bf16).  The final
        // o = O / l is the same for any choice of reference.
        constexpr float RESCALE_LOG2 = 8.f;
        const int quad = warp & 3;                       // TMEM lanes this warp may access
        const int r = quad * 32 + lane;                  // row = TMEM lane
        const int tt = r / p.H, h = r % p.H;
        const int i = i0 + tt;
        const bool row_ok = tt < p.T && i < p.n_q;
        const bool warp_idle = __all_sync(FULL, !row_ok);
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float sl2 = p.scale_log2;

        // Dense modes: the keys this row sees, as an absolute interval [ka, kb).
        long long ka = 0, kb = 0;
        if (MODE != 0 && row_ok) {
            const long long t = p.q_pos0 + i;
            if (MODE == 1) {
                const long long nv = (t + 1) / p.m;
                ka = r_lo;
                kb = nv < r_hi ? nv : r_hi;
            } else {
                const long long lo = t - p.window + 1;
                ka = lo > r_lo ? lo : r_lo;
                kb = (t + 1) < r_hi ? (t + 1) : r_hi;
            }
        }

        float m_ref = -INFINITY, l_run = 0.f;
        bool ok = true;
        if (MODE == 0 && n_tiles > 0) ok = __all_sync(FULL, mbar_wait(bar_list, 0, abort_flag));
        for (int j = 0; ok && j < n_tiles; ++j) {
            const int sb = j % SBUFS;
            const bool w = mbar_wait(&s_full[sb], (j / SBUFS) & 1, abort_flag);
            if (!__all_sync(FULL, w)) { ok = false; break; }
            tc_fence_after();
            if (!warp_idle) {
                // validity of column c: mode 0 bit (c / 4) of mask word (c % 4);
                // dense modes c in [lo_c, hi_c)
                uint32_t mk[4] = {0u, 0u, 0u, 0u};
                int lo_c = 0, hi_c = 0;
                if (MODE == 0) {
                    // bit l of word u: entry 4l + u of the tile is a valid index
                    const int4 q4 = reinterpret_cast<const int4*>(sidx + j * KT)[lane];
                    mk[0] = __ballot_sync(FULL, q4.x >= 0);
                    mk[1] = __ballot_sync(FULL, q4.y >= 0);
                    mk[2] = __ballot_sync(FULL, q4.z >= 0);
                    mk[3] = __ballot_sync(FULL, q4.w >= 0);
                    if (!row_ok) mk[0] = mk[1] = mk[2] = mk[3] = 0u;
                } else {
                    const long long kbase = r_lo + (long long)j * KT;
                    const long long a = ka - kbase, e = kb - kbase;
                    lo_c = (int)(a < 0 ? 0 : (a > KT ? KT : a));
                    hi_c = (int)(e < 0 ? 0 : (e > KT ? KT : e));
                }
                const uint32_t s_addr = tmem + lane_base + S_COL + sb * KT;
                float sum = 0.f;
                // the rescale of O when this tile's maximum moves the reference;
                // false on a timeout
                auto move_reference = [&](float mx) -> bool {
                    const bool move = mx > m_ref + RESCALE_LOG2;
                    const float m_new = move ? mx : m_ref;
                    if (__any_sync(FULL, move && m_ref != -INFINITY)) {
                        // O holds P_0..P_{j-1} V against the old reference: wait
                        // for P_{j-1} V_{j-1}, then rescale the rows that moved
                        const bool w2 = mbar_wait(o_full, (j - 1) & 1, abort_flag);
                        if (!__all_sync(FULL, w2)) return false;
                        tc_fence_after();
                        const float f = (move && m_ref != -INFINITY) ? ex2_approx(m_ref - m_new) : 1.f;
                        const uint32_t o_addr = tmem + lane_base + O_COL;
                        // 16 columns at a time: the tile's scores stay live meanwhile
#pragma unroll
                        for (int q = 0; q < D / 16; ++q) {
                            uint32_t ov[16];
                            tmem_ld16(o_addr + 16 * q, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int u = 0; u < 16; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * f);
                            tmem_st16(o_addr + 16 * q, ov);
                        }
                        l_run *= f;
                    }
                    m_ref = m_new;
                    return true;
                };
                if constexpr (R::SPARSE || SBUFS == 1) {
                    // two passes over 32-column chunks of S: the row maximum,
                    // then the exponentials (a chunk's P overwrites S columns
                    // already read: P of chunk q lands in columns 16q .. 16q+15);
                    // the register budget of a 512-thread CTA or of two CTAs an SM
                    const bool all_full = R::SPARSE ? __all_sync(FULL, row_ok && (mk[0] & mk[1] & mk[2] & mk[3]) == FULL)
                                                    : __all_sync(FULL, lo_c == 0 && hi_c == KT);
                    auto load_chunk = [&](int q, float (&v)[32]) {
                        tmem_ld32(s_addr + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                        tmem_ld_wait();
                        if (!all_full) {
#pragma unroll
                            for (int u = 0; u < 32; ++u) {
                                const int c = 32 * q + u;
                                const bool valid = R::SPARSE ? ((mk[c & 3] >> (c >> 2)) & 1u) != 0u
                                                             : (unsigned)(c - lo_c) < (unsigned)(hi_c - lo_c);
                                v[u] = valid ? v[u] : -INFINITY;
                            }
                        }
                    };
                    float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
                    for (int q = 0; q < KT / 32; ++q) {
                        float v[32];
                        load_chunk(q, v);
#pragma unroll
                        for (int u = 0; u < 32; u += 4) {
                            a0 = fmax3(a0, v[u], v[u + 1]);
                            a1 = fmax3(a1, v[u + 2], v[u + 3]);
                        }
                    }
                    // scores are raw dot products; the positive scale commutes with max
                    if (!move_reference(fmaxf(a0, a1) * sl2)) { ok = false; break; }
                    const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
                    for (int q = 0; q < KT / 32; ++q) {
                        float v[32];
                        load_chunk(q, v);
                        uint32_t pk[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float p0 = ex2_approx(fmaf(v[2 * u], sl2, neg_m));
                            const float p1 = ex2_approx(fmaf(v[2 * u + 1], sl2, neg_m));
                            sum += p0 + p1;
                            pk[u] = pack_bf16x2(p0, p1);
                        }
                        tmem_st16(s_addr + 16 * q, pk);
                    }
                } else {
                    float sv[KT];
#pragma unroll
                    for (int q = 0; q < KT / 32; ++q) tmem_ld32(s_addr + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * q]));
                    tmem_ld_wait();
                    // masked columns become -inf; a tile valid for every row of the
                    // warp (the common case) skips the masking
                    const bool full_row = lo_c == 0 && hi_c == KT;
                    if (!__all_sync(FULL, full_row)) {
#pragma unroll
                        for (int c = 0; c < KT; ++c)
                            sv[c] = ((unsigned)(c - lo_c) < (unsigned)(hi_c - lo_c)) ? sv[c] : -INFINITY;
                    }
                    float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                    for (int c = 0; c < KT; c += 8) {
                        a0 = fmax3(a0, sv[c], sv[c + 1]);
                        a1 = fmax3(a1, sv[c + 2], sv[c + 3]);
                        a2 = fmax3(a2, sv[c + 4], sv[c + 5]);
                        a3 = fmax3(a3, sv[c + 6], sv[c + 7]);
                    }
                    // scores are raw dot products; the positive scale commutes with max
                    if (!move_reference(fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * sl2)) { ok = false; break; }
                    const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
                    for (int q = 0; q < KT / 32; ++q) {
                        uint32_t pk[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float p0 = ex2_approx(fmaf(sv[32 * q + 2 * u], sl2, neg_m));
                            const float p1 = ex2_approx(fmaf(sv[32 * q + 2 * u + 1], sl2, neg_m));
                            sum += p0 + p1;
                            pk[u] = pack_bf16x2(p0, p1);
                        }
                        // P columns 16q..16q+15 overwrite S columns already read
                        tmem_st16(s_addr + 16 * q, pk);
                    }
                }
                tmem_st_wait();
                l_run += sum;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }

        if (ok && n_tiles > 0) {
            // every MMA of the CTA has retired (a single-use barrier: the
            // per-tile o_full phases cannot tell the last two tiles apart here)
            const bool w = mbar_wait(bar_mma_done, 0, abort_flag);
            ok = __all_sync(FULL, w);
            if (ok) tc_fence_after();
        }
        if (ok && !warp_idle) {
            const long long grow = ((long long)b * p.n_q + i) * p.H + h;   // (b, token, head)
            const uint32_t o_addr = tmem + lane_base + O_COL;
            const bool split_out = p.n_splits > 1;
            const float inv = (!split_out && l_run > 0.f) ? 1.f / l_run : (split_out ? 1.f : 0.f);
            const long long prow = (long long)split * p.B * p.n_q * p.H + grow;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t ov[32];
                if (n_tiles > 0) {
                    tmem_ld32(o_addr + 32 * q, ov);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) ov[u] = 0u;
                }
                if (!row_ok) continue;
                if (!split_out) {
                    uint4* op = reinterpret_cast<uint4*>(p.out + grow * D + 32 * q);
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w4;
                        w4.x = pack_bf16x2(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
                        w4.y = pack_bf16x2(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
                        w4.z = pack_bf16x2(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
                        w4.w = pack_bf16x2(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
                        op[c / 8] = w4;
                    }
                } else {
                    float4* po = reinterpret_cast<float4*>(p.part_o + prow * D + 32 * q);
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        po[c / 4] = make_float4(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1]),
                                                __uint_as_float(ov[c + 2]), __uint_as_float(ov[c + 3]));
                }
            }
            if (row_ok) {
                if (!split_out) {
                    if (p.lse) p.lse[grow] = l_run > 0.f ? (m_ref + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
                } else {
                    p.part_ml[2 * prow] = l_run > 0.f ? m_ref : -INFINITY;
                    p.part_ml[2 * prow + 1] = l_run;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == R::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

bool attn_tc_supported(int H, int D) { return (H == 64 || H == 128) && D == atc::D; }

int attn_tc_tokens_per_cta(int mode, int H) { return mode == 0 ? 1 : atc::ROWS / H; }

int attn_tc_q_box_rows(int mode, int H) { return (mode == 0 && H == 64) ? 64 : 128; }

template <int MODE, int STAGES, int QROWS, int SBUFS = 2>
static void launch_one(dim3 grid, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const AttnTcParams& p, cudaStream_t s)
{
    auto kern = attn_tc_kernel<MODE, STAGES, QROWS, SBUFS>;
    constexpr int smem = atc::Cfg<MODE, STAGES, QROWS>::SMEM;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    (void)launch_pdl(kern, dim3(grid), dim3(atc::Roles<MODE>::THREADS), smem, s, tq, tk, tv, p);
}

cudaError_t launch_attn_tc(int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnTcParams& p, cudaStream_t s)
{
    if ((long long)p.B * p.n_q == 0) return cudaSuccess;
    const int n_groups = (p.n_q + p.T - 1) / p.T;
    dim3 grid((unsigned)(n_groups * p.n_splits), (unsigned)p.B);
    if (mode == 0) {
        if (p.H == 64) launch_one<0, 3, 64>(grid, tq, tk, tv, p, s);
        else launch_one<0, 2, 128>(grid, tq, tk, tv, p, s);
    } else {
        // dense modes: short key sets (the stack's SWA windows and HCA prefixes)
        // take the small configuration, two CTAs an SM
        long long set_max = mode == 2 ? p.window + p.T - 1 : std::min<long long>(p.N_kv, (p.q_pos0 + p.n_q) / p.m);
        if (p.n_splits > 1) set_max = std::min<long long>(set_max, p.split_len);
        const bool small = (set_max + atc::KT - 1) / atc::KT <= atc::SMALL_MAX_TILES;
        if (mode == 1) {
            if (small) launch_one<1, 1, 128, 1>(grid, tq, tk, tv, p, s);
            else launch_one<1, 3, 128>(grid, tq, tk, tv, p, s);
        } else {
            if (small) launch_one<2, 1, 128, 1>(grid, tq, tk, tv, p, s);
            else launch_one<2, 3, 128>(grid, tq, tk, tv, p, s);
        }
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.n_splits == 1) return e;
    AttnArgsT<__nv_bfloat16> a{};
    a.out = p.out;
    a.lse = p.lse;
    a.part_o = p.part_o;
    a.part_ml = p.part_ml;
    a.B = p.B;
    a.n_q = p.n_q;
    a.n_splits = p.n_splits;
    return launch_attn_combine(a, p.H, atc::D, s);
}

}  // namespace csa
