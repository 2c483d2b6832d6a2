// Merge of split-KV partials: a query row's key set, cut into n_splits
// slices, leaves per slice the unnormalised o_s (against the slice's
// reference maximum m_s, base-2 domain) and l_s.  In split order:
//     M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  o = sum_s o_s 2^(m_s - M) / L,
// lse = (M + log2 L) ln 2 (-inf and o = 0 when every slice is empty).
// Loads go through L2 (the partials may have been written by other CTAs of
// the running kernel).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace csa {

// One (row * H + h, 8 channels c .. c+7) item.
template <typename TIO>
__device__ __forceinline__ void merge_split_partials(const AttnArgsT<TIO>& a, int H, int D, long long rh, int c)
{
    const long long stride = (long long)a.B * a.n_q * H;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml);   // (m, l) per split and row
    // Splits are merged SU at a time with all their loads in flight: every
    // split of a batch is weighted against the running maximum M (the
    // batch's maximum folded in first; earlier sums rescaled).
    constexpr int SU = 8;
    float M = -INFINITY, L = 0.f, o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = 0.f;
    for (int s0 = 0; s0 < a.n_splits; s0 += SU) {
        float2 mv[SU];
        float4 pa[SU], pb[SU];
#pragma unroll
        for (int u = 0; u < SU; ++u) {
            const int sp = s0 + u;
            if (sp < a.n_splits) {
                const long long r = sp * stride + rh;
                mv[u] = __ldcg(ml + r);
                const float4* po = reinterpret_cast<const float4*>(a.part_o + r * D + c);
                pa[u] = __ldcg(po);
                pb[u] = __ldcg(po + 1);
            } else {
                mv[u] = make_float2(-INFINITY, 0.f);
                pa[u] = pb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mb = M;
#pragma unroll
        for (int u = 0; u < SU; ++u) Mb = fmaxf(Mb, mv[u].x);
        if (Mb == -INFINITY) continue;            // every split so far is empty
        const float rs = exp2f(M - Mb);           // 0 while M = -inf
        L *= rs;
#pragma unroll
        for (int v = 0; v < 8; ++v) o[v] *= rs;
#pragma unroll
        for (int u = 0; u < SU; ++u) {
            const float w = exp2f(mv[u].x - Mb);  // 0 for empty splits (m = -inf)
            L = fmaf(mv[u].y, w, L);
            o[0] = fmaf(pa[u].x, w, o[0]);
            o[1] = fmaf(pa[u].y, w, o[1]);
            o[2] = fmaf(pa[u].z, w, o[2]);
            o[3] = fmaf(pa[u].w, w, o[3]);
            o[4] = fmaf(pb[u].x, w, o[4]);
            o[5] = fmaf(pb[u].y, w, o[5]);
            o[6] = fmaf(pb[u].z, w, o[6]);
            o[7] = fmaf(pb[u].w, w, o[7]);
        }
        M = Mb;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] *= inv;
    Vec8<TIO>::store(a.out + rh * D + c, o);
    if (a.lse && c == 0) a.lse[rh] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace csa
