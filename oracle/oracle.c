/*
 * CPU oracle for DeepSeek-V4 hybrid long-context attention (CSA / HCA / SWA).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path never
 * calls it, and it shares no code, header, table or helper with the CUDA
 * kernels.
 *
 * Plain, slow, obviously correct: scalar loops, fp64 accumulation, no tiling,
 * no fusion.  Parallelism is only over independent output rows (OpenMP), which
 * does not change any result.  Where a floating-point value decides an
 * integer (a quantised code, the ranking behind the top-k), the decision is
 * taken on an fp32 value, the precision the GPU kernels decide in.
 *
 * Sources:
 *  - "DeepSeek V4 技术解读" (takeshell.com), §2.1 CSA: every m tokens' KV entries
 *    are merged by weighted aggregation into one entry (length n/m); a
 *    Lightning Indexer scores each query's indexer queries against the
 *    compressed entries and keeps the top-k; core attention runs only over the
 *    k selected entries.  m=4, 64 indexer heads of dim 128, k=1024.
 *  - same page, §2.2 HCA: compression at m'=128, then full attention over all
 *    compressed entries with no selection.
 *  - same page, §2.3: the first two layers are pure sliding-window attention.
 *  - same page, §五: FP4 (E2M1) -> FP8 (E4M3) dequantisation, lossless while the
 *    spread of block scale factors stays within a threshold.
 * Points those passages leave open are fixed as stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                           */
/* E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;   */
/* exponent field 0 is subnormal (m/8 * 2^-6); 0x7F/0xFF are NaN; no inf.    */
/* Largest finite value 1.75 * 2^8 = 448.                                    */
/* E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0  */
/* is subnormal (m/2 * 2^0).  Values 0, 0.5, 1, 1.5, 2, 3, 4, 6.             */
/* ------------------------------------------------------------------------ */

ORC_API double orc_e4m3_value(unsigned c)
{
    c &= 0xFFu;
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, mt = c & 7;
    double v;
    if (e == 0xF && mt == 7) return NAN;
    if (e == 0) v = ldexp((double)mt / 8.0, -6);
    else v = ldexp(1.0 + (double)mt / 8.0, e - 7);
    return s ? -v : v;
}

ORC_API double orc_e2m1_value(unsigned c)
{
    c &= 0xFu;
    int s = (c >> 3) & 1, e = (c >> 1) & 3, mt = c & 1;
    double v;
    if (e == 0) v = 0.5 * mt;
    else v = ldexp(1.0 + 0.5 * mt, e - 1);
    return s ? -v : v;
}

/* Round |a| to the format's grid, ties to even.  q = value of one unit in the
 * last mantissa place of a's binade (clamped to the subnormal quantum). */
static double round_to_grid(double a, int min_exp, int mant_bits)
{
    int ex;
    frexp(a, &ex);                      /* a = f * 2^ex, f in [0.5, 1) */
    int fl = ex - 1;                    /* floor(log2 a) for a > 0 */
    if (fl < min_exp) fl = min_exp;
    double q = ldexp(1.0, fl - mant_bits);
    return nearbyint(a / q) * q;        /* default rounding mode: to even */
}

/* E4M3 encode with round-to-nearest-even and saturation to +-448. */
ORC_API unsigned orc_e4m3_encode(float y)
{
    if (isnan(y)) return 0x7F;
    unsigned s = signbit(y) ? 0x80u : 0u;
    double a = fabs((double)y);
    if (a == 0.0) return s;
    double r = round_to_grid(a, -6, 3);
    if (r >= 448.0) return s | 0x7E;
    if (r == 0.0) return s;
    if (r < ldexp(1.0, -6)) {            /* subnormal: r = mt * 2^-9 */
        unsigned mt = (unsigned)(r / ldexp(1.0, -9));
        return s | mt;
    }
    int ex;
    double f = frexp(r, &ex);           /* r = f * 2^ex, f in [0.5,1) */
    unsigned e = (unsigned)(ex - 1 + 7);
    unsigned mt = (unsigned)((2.0 * f - 1.0) * 8.0);
    return s | (e << 3) | mt;
}

/* E2M1 encode with round-to-nearest-even and saturation to +-6. */
ORC_API unsigned orc_e2m1_encode(float y)
{
    unsigned s = signbit(y) ? 0x8u : 0u;
    double a = fabs((double)y);
    if (isnan(y)) return 0x7;           /* no NaN in E2M1: saturate */
    if (a == 0.0) return s;
    double r = round_to_grid(a, 0, 1);
    if (r > 6.0) r = 6.0;
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    for (unsigned i = 0; i < 8; ++i)
        if (grid[i] == r) return s | i;
    return s | 7u;                      /* unreachable for finite input */
}

ORC_API void orc_e4m3_decode_array(int64_t n, const uint8_t* c, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (float)orc_e4m3_value(c[i]);
}

ORC_API void orc_e4m3_encode_array(int64_t n, const float* y, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(y[i]);
}

ORC_API void orc_e2m1_encode_array(int64_t n, const float* y, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(y[i]);
}

/* ------------------------------------------------------------------------ */
/* a1: KV compression ("DeepSeek V4 技术解读" §2.1 / §2.2).                    */
/* Block j of m tokens becomes one entry: out[j] = sum_i w_i * x[j*m + i],  */
/* with w = softmax over the block of one scalar logit per token (the spec's */
/* reading of "weighted aggregation").  Only closed blocks: N_c = n / m.    */
/* ------------------------------------------------------------------------ */
ORC_API void orc_compress(int B, int n, int m, int d, const float* logits,
                          const float* x, double* out)
{
    int Nc = n / m;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < Nc; ++j) {
            const float* lg = logits + (int64_t)b * n + (int64_t)j * m;
            double mx = -INFINITY;
            for (int i = 0; i < m; ++i) if (lg[i] > mx) mx = lg[i];
            double den = 0.0;
            for (int i = 0; i < m; ++i) den += exp((double)lg[i] - mx);
            double* o = out + ((int64_t)b * Nc + j) * d;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            for (int i = 0; i < m; ++i) {
                double w = exp((double)lg[i] - mx) / den;
                const float* xr = x + ((int64_t)b * n + (int64_t)j * m + i) * d;
                for (int c = 0; c < d; ++c) o[c] += w * (double)xr[c];
            }
        }
}

/* a1 variant: per-channel compression weights -- a reading of "weighted
 * aggregation" (加权聚合, "DeepSeek V4 技术解读" §2.1) in which every channel
 * c carries its own logit per token: out[j][c] = sum_i w_{j,i,c} x[jm+i][c],
 * w_{j,.,c} = softmax over the block of logits[jm+i][c].  logits: [B, n, d]. */
ORC_API void orc_compress_per_channel(int B, int n, int m, int d, const float* logits,
                                      const float* x, double* out)
{
    int Nc = n / m;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < Nc; ++j)
            for (int c = 0; c < d; ++c) {
                const float* lg = logits + ((int64_t)b * n + (int64_t)j * m) * d + c;
                double mx = -INFINITY;
                for (int i = 0; i < m; ++i) if (lg[(int64_t)i * d] > mx) mx = lg[(int64_t)i * d];
                double den = 0.0;
                for (int i = 0; i < m; ++i) den += exp((double)lg[(int64_t)i * d] - mx);
                double acc = 0.0;
                for (int i = 0; i < m; ++i) {
                    double w = exp((double)lg[(int64_t)i * d] - mx) / den;
                    acc += w * (double)x[((int64_t)b * n + (int64_t)j * m + i) * d + c];
                }
                out[((int64_t)b * Nc + j) * d + c] = acc;
            }
}

/* Per-row E4M3 quantisation of compressed indexer keys (the compression
 * epilogue).  scale = amax / 448, code = E4M3(x * (448 / amax)), all in fp32;
 * a row with amax = 0 gets scale 1 and zero codes. */
ORC_API void orc_quant_e4m3_rows(int64_t rows, int d, const float* x,
                                 uint8_t* codes, float* scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * d;
        float amax = 0.0f;
        for (int c = 0; c < d; ++c) { float a = fabsf(xr[c]); if (a > amax) amax = a; }
        float inv = 1.0f, sc = 1.0f;
        if (amax > 0.0f) { inv = 448.0f / amax; sc = amax / 448.0f; }
        for (int c = 0; c < d; ++c) {
            float y = xr[c] * inv;            /* one fp32 rounding */
            codes[r * d + c] = (uint8_t)orc_e4m3_encode(y);
        }
        scale[r] = sc;
    }
}

/* Per-32-element E2M1 quantisation with an E4M3 block scale (the compression
 * epilogue for FP4 indexer keys).  sc = E4M3(amax / 6), raised to the smallest
 * positive E4M3 value if it rounds to zero; code = E2M1(x / sc) in fp32.
 * Packing: element 2i in the low nibble, element 2i+1 in the high nibble. */
ORC_API void orc_quant_e2m1_blocks(int64_t rows, int d, const float* x,
                                   uint8_t* packed, uint8_t* sc_codes)
{
    int nb = d / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int blk = 0; blk < nb; ++blk) {
            const float* xr = x + r * d + blk * 32;
            float amax = 0.0f;
            for (int c = 0; c < 32; ++c) { float a = fabsf(xr[c]); if (a > amax) amax = a; }
            float t = amax / 6.0f;
            unsigned scc = orc_e4m3_encode(t);
            if ((scc & 0x7F) == 0) scc = 0x01;
            float sc = (float)orc_e4m3_value(scc);
            sc_codes[r * nb + blk] = (uint8_t)scc;
            for (int c = 0; c < 32; c += 2) {
                float y0 = xr[c] / sc, y1 = xr[c + 1] / sc;
                unsigned e0 = orc_e2m1_encode(y0), e1 = orc_e2m1_encode(y1);
                packed[r * (d / 2) + (blk * 32 + c) / 2] = (uint8_t)(e0 | (e1 << 4));
            }
        }
    }
}

/* FP4 -> FP8 dequantisation ("DeepSeek V4 技术解读" §五).  Reading: per row,
 * S = 2^(floor(log2(max_b sc_b)) - 5), a power of two; each element becomes
 * x8 = E4M3(e * sc_b / S) with one rounding, and the row's scale is S.  The
 * product e * sc_b and the division by S are exact in fp32, so the only
 * rounding is the E4M3 encode: the conversion is lossless exactly when every
 * e * sc_b / S lies on the E4M3 grid.  Returns the number of elements that
 * were rounded. */
ORC_API int64_t orc_fp4_to_e4m3(int64_t rows, int d, const uint8_t* packed,
                                const uint8_t* sc_codes, uint8_t* x8, float* S)
{
    int nb = d / 32;
    int64_t rounded = 0;
#pragma omp parallel for schedule(static) reduction(+:rounded)
    for (int64_t r = 0; r < rows; ++r) {
        float mx = 0.0f;
        for (int blk = 0; blk < nb; ++blk) {
            float v = (float)orc_e4m3_value(sc_codes[r * nb + blk]);
            if (v > mx) mx = v;
        }
        int ex;
        frexp((double)mx, &ex);
        double Sd = ldexp(1.0, (ex - 1) - 5);
        S[r] = (float)Sd;
        for (int c = 0; c < d; ++c) {
            unsigned byte = packed[r * (d / 2) + c / 2];
            unsigned e = (c & 1) ? (byte >> 4) : (byte & 0xF);
            float sc = (float)orc_e4m3_value(sc_codes[r * nb + c / 32]);
            float prod = (float)orc_e2m1_value(e) * sc;
            float y = prod / (float)Sd;
            unsigned code = orc_e4m3_encode(y);
            x8[r * d + c] = (uint8_t)code;
            if (orc_e4m3_value(code) != (double)y) ++rounded;
        }
    }
    return rounded;
}

/* ------------------------------------------------------------------------ */
/* Visibility: compressed entry j is visible to the query at absolute        */
/* position t iff its block is closed, (j+1)*m - 1 <= t.                     */
/* ------------------------------------------------------------------------ */
static int64_t n_visible(int64_t t, int m, int64_t Nc)
{
    int64_t v = (t + 1) / m;
    return v < Nc ? v : Nc;
}

/* a2: Lightning-Indexer scores ("DeepSeek V4 技术解读" §2.1; 64 heads x 128).
 * s(t, j) = sum_h sq(t,h) * sk(j) * <q(t,h), k(j)>, heads summed in order
 * h = 0..H_I-1, for j < nv(t).  q and k hold the decoded stored values; the
 * scale arrays may be NULL (scale 1).  Entries j >= nv(t) are set to NaN.
 * Variant reading of the page's "similarity" (§8 f3): with relu, each head's
 * term uses max(<q, k>, 0) (the scales are positive, so this is the ReLU of
 * the scaled dot product), and with head_w ([B, n_q, H_I]) each head's term
 * is multiplied by w(t, h): s = sum_h w(t,h) * sq * sk * ReLU(<q, k>).
 * rows: NULL for all B*n_q rows, else n_rows flat indices b*n_q + i.
 * out64 gets the fp64 score, out32 (optional) the same value rounded to fp32,
 * the value the ranking uses. */
ORC_API void orc_index_scores(int B, int n_q, int64_t q_pos0, int m, int Nc,
                              int HI, int dI, const float* q, const float* q_scale,
                              const float* k, const float* k_scale,
                              const float* head_w, int relu,
                              int n_rows, const int64_t* rows,
                              double* out64, float* out32)
{
    int64_t R = rows ? n_rows : (int64_t)B * n_q;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t r = 0; r < R; ++r)
        for (int64_t j = 0; j < Nc; ++j) {
            int64_t flat = rows ? rows[r] : r;
            int64_t b = flat / n_q, i = flat % n_q;
            int64_t nv = n_visible(q_pos0 + i, m, Nc);
            const float* qt = q + flat * HI * dI;
            double s = NAN;
            if (j < nv) {
                const float* kr = k + (b * Nc + j) * dI;
                double sk = k_scale ? (double)k_scale[b * Nc + j] : 1.0;
                s = 0.0;
                for (int h = 0; h < HI; ++h) {
                    double dot = 0.0;
                    for (int c = 0; c < dI; ++c)
                        dot += (double)qt[h * dI + c] * (double)kr[c];
                    double sq = q_scale ? (double)q_scale[flat * HI + h] : 1.0;
                    if (relu && dot < 0.0) dot = 0.0;
                    double term = sq * sk * dot;
                    if (head_w) term *= (double)head_w[flat * HI + h];
                    s += term;
                }
            }
            if (out64) out64[r * Nc + j] = s;
            if (out32) out32[r * Nc + j] = (float)s;
        }
}

/* a3: top-k ("DeepSeek V4 技术解读" §2.1: keep the k highest-scoring entries).
 * Ranking by (fp32 score descending, index ascending), -0 counted as +0.  The
 * first min(k, len) are returned in ascending index order, -1 padded. */
typedef struct { float s; int32_t j; } scored_t;

static int cmp_scored(const void* a, const void* b)
{
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int cmp_i32(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

ORC_API void orc_topk(int n_rows, const int64_t* lens, int64_t row_stride, int k,
                      const float* scores, int32_t* out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
        int64_t L = lens[r];
        scored_t* v = (scored_t*)malloc(sizeof(scored_t) * (L > 0 ? L : 1));
        for (int64_t j = 0; j < L; ++j) {
            float s = scores[(int64_t)r * row_stride + j];
            if (s == 0.0f) s = 0.0f;        /* -0 -> +0 */
            v[j].s = s;
            v[j].j = (int32_t)j;
        }
        qsort(v, (size_t)L, sizeof(scored_t), cmp_scored);
        int64_t c = L < k ? L : k;
        int32_t* o = out + (int64_t)r * k;
        for (int64_t i = 0; i < c; ++i) o[i] = v[i].j;
        qsort(o, (size_t)c, sizeof(int32_t), cmp_i32);
        for (int64_t i = c; i < k; ++i) o[i] = -1;
        free(v);
    }
}

/* a4 / a5 / a6: attention of H query heads over one shared KV head.
 * o(t,h) = sum_j softmax_j(tau * <q(t,h), K[j]>) V[j] over the key set of t,
 * lse(t,h) = log sum_j exp(tau * <q, K[j]>).  Two passes (max, then sum), fp64.
 * An empty key set gives o = 0 and lse = -inf.
 *   mode 0, sparse (CSA core attention, §2.1): the set is idx[b, i, :],
 *           entries < 0 are padding.
 *   mode 1, closed blocks (HCA, §2.2): j < nv(t) = min(floor((t+1)/m), N_kv).
 *   mode 2, window (§2.3): max(0, t-W+1) <= j <= min(t, N_kv-1).
 * q: [B, n_q, H, d]; K, V: [B, N_kv, H_kv, d] (H_kv KV heads; query head h
 * reads KV head h / (H / H_kv) -- H_kv = 1 is the shared head of the MLA
 * reading, H_kv > 1 the GQA / MHA variant readings); idx: [B, n_q, k].
 * out: [R, H, d], lse: [R, H] for the R selected rows. */
ORC_API void orc_attention(int B, int n_q, int H, int H_kv, int d, int64_t Nkv,
                           const float* q, const float* K, const float* V,
                           double tau, int mode, int64_t q_pos0, int m,
                           int64_t window, const int32_t* idx, int k,
                           int n_rows, const int64_t* rows,
                           double* out, double* lse)
{
    int64_t R = rows ? n_rows : (int64_t)B * n_q;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r)
        for (int h = 0; h < H; ++h) {
            int64_t flat = rows ? rows[r] : r;
            int64_t b = flat / n_q, i = flat % n_q, t = q_pos0 + i;
            int64_t cnt, lo = 0;
            const int32_t* sel = NULL;
            if (mode == 0) { sel = idx + flat * k; cnt = k; }
            else if (mode == 1) { cnt = n_visible(t, m, Nkv); }
            else {
                lo = t - window + 1; if (lo < 0) lo = 0;
                int64_t hi = t < Nkv - 1 ? t : Nkv - 1;
                cnt = hi >= lo ? hi - lo + 1 : 0;
            }
            const int64_t hk = h / (H / H_kv);    /* this head's KV head */
            const float* qh = q + (flat * H + h) * d;
            double* o = out + (r * H + h) * d;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            double mx = -INFINITY;
            for (int64_t e = 0; e < cnt; ++e) {
                int64_t j = sel ? sel[e] : lo + e;
                if (j < 0) continue;
                if (j >= Nkv) { mx = NAN; break; }
                const float* kr = K + ((b * Nkv + j) * H_kv + hk) * d;
                double s = 0.0;
                for (int c = 0; c < d; ++c) s += (double)qh[c] * (double)kr[c];
                s *= tau;
                if (s > mx) mx = s;
            }
            if (isnan(mx)) {
                for (int c = 0; c < d; ++c) o[c] = NAN;
                lse[r * H + h] = NAN;
                continue;
            }
            if (mx == -INFINITY) { lse[r * H + h] = -INFINITY; continue; }
            double den = 0.0;
            for (int64_t e = 0; e < cnt; ++e) {
                int64_t j = sel ? sel[e] : lo + e;
                if (j < 0) continue;
                const float* kr = K + ((b * Nkv + j) * H_kv + hk) * d;
                const float* vr = V + ((b * Nkv + j) * H_kv + hk) * d;
                double s = 0.0;
                for (int c = 0; c < d; ++c) s += (double)qh[c] * (double)kr[c];
                double p = exp(s * tau - mx);
                den += p;
                for (int c = 0; c < d; ++c) o[c] += p * (double)vr[c];
            }
            for (int c = 0; c < d; ++c) o[c] /= den;
            lse[r * H + h] = mx + log(den);
        }
}

ORC_API int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
