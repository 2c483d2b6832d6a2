// Launchers of the device kernels, called by the C-ABI layer (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "../../include/csa.h"

namespace csa {

// Records the thread's last-error message (api.cu) and returns st.
csa_status_t report(csa_status_t st, const char* msg);

// ---- compression ----
// out_kind: 0 f32, 1 bf16, 2 e4m3 (+ fp32 row scale), 3 e2m1 (+ e4m3 block scales)
cudaError_t launch_compress(int B, int n, int m, int d, const float* logits, const void* x, bool x_bf16,
                            void* out, int out_kind, void* out_scale, int num_sms, cudaStream_t s);
// Per-channel compression weights: logits [B, n, d] (one logit per token and
// channel); out_kind as above.
cudaError_t launch_compress_per_channel(int B, int n, int m, int d, const float* logits, const void* x, bool x_bf16,
                                        void* out, int out_kind, void* out_scale, cudaStream_t s);
// All streams in one launch, for short blocks (4 <= m <= 32, m and n multiples
// of 4, one tile entry within the stage budget); out_kind 0 f32, 1 bf16,
// 2 e4m3, 3 e2m1.
bool compress_tiles_supported(int n, int m, int n_streams, const int* dim, const bool* x_bf16);
cudaError_t launch_compress_tiles(int B, int n, int m, int n_streams, const float* logits, const void* const* x,
                                  const bool* x_bf16, const int* dim, void* const* out, const int* out_kind,
                                  void* const* out_scale, int num_sms, cudaStream_t s);

// Query positions: query i of sequence b sits at at(b) + i, where at(b) is
// q_pos0, or lens[b] + off when per-sequence token counts (a device array)
// are given.  at() with lens reads device memory: device code only.
struct QPos {
    long long q_pos0 = 0;
    const long long* lens = nullptr;
    long long off = 0;
    QPos() = default;
    QPos(long long p) : q_pos0(p) {}   // NOLINT: a single start for every sequence
    QPos(const long long* l, long long o) : lens(l), off(o) {}
    __device__ __forceinline__ long long at(long long b) const { return lens ? lens[b] + off : q_pos0; }
    // the same positions shifted by i0 queries (a chunk of rows)
    QPos shifted(long long i0) const { QPos q = *this; q.q_pos0 += i0; q.off += i0; return q; }
};

// ---- streaming decode state ----
constexpr int DECODE_MAX_M = 128;     // longest block (HCA's m' = 128)
constexpr int DECODE_MAX_DIM = 256;
struct DecodeAppendArgs {
    int B, m, d, d_I;
    long long N_cap;                  // entries each sequence's caches hold
    const float* logit_new;           // [B]
    const void* k_new;                // [B, d]   (input dtype)
    const void* v_new;                // [B, d]
    const void* ik_new;               // [B, d_I]
    float* st_logit;                  // [B, m]   the open block, raw tokens
    void* st_k;                       // [B, m, d]
    void* st_v;                       // [B, m, d]
    void* st_ik;                      // [B, m, d_I]
    long long* lens;                  // [B] tokens appended so far (advanced)
    void* k_c;                        // [B, N_cap, d]
    void* v_c;                        // [B, N_cap, d]
    int kv_kind;                      // 0 fp32, 1 bf16
    void* ik_c;                       // [B, N_cap, d_I] (E2M1: d_I / 2 bytes a row)
    void* ik_scale;                   // E4M3: fp32 [B, N_cap]; E2M1: E4M3 [B, N_cap, d_I / 32]
    int ik_kind;                      // 0 fp32, 1 bf16, 2 e4m3, 3 e2m1
};
cudaError_t launch_decode_append(const DecodeAppendArgs& a, bool x_bf16, cudaStream_t s);

// ---- top-k ----
constexpr int TOPK_MAX_SINGLE = 32768;   // entries one CTA selects from (keys in smem)
constexpr int TOPK_MAX_ROW = 524288;     // longest row (the select kernel's bitmaps)
struct TopkPlan { int chunk; int n_chunks; };
TopkPlan topk_plan(int N_c, int k);
bool topk_supported(int N_c, int k);
// rows * chunks of a long row fit one grid dimension (INT_MAX CTAs)
bool topk_rows_ok(long long rows, int N_c, int k);
size_t topk_workspace_bytes(long long rows, int N_c, int k);
// wmax (optional, rows longer than one CTA's capacity): per row, the
// largest score key of every run of 32 consecutive entries (wmax_ld words a
// row), written by the decode indexer; the collection then takes its
// threshold from them instead of from a sample of the row.
// scores: fp32, or bf16 when scores_bf16 (selection on the stored values).
// counters_clear: the rows' counters (topk_row_counters) were cleared by the
// kernel before (the fused route's indexer), so no memset is issued.
cudaError_t launch_topk(const void* scores, bool scores_bf16, long long ld, int B, int n_q_rows, QPos q_pos0,
                        int m, int N_c, int k, int32_t* out, long long out_b_stride, void* ws,
                        cudaStream_t s, const uint32_t* wmax = nullptr, int wmax_ld = 0,
                        bool counters_clear = false);
// The long-row route's per-row counters (one word a row, at the start of the
// top-k workspace), which every long-row selection needs cleared first.
uint32_t* topk_row_counters(void* ws);
bool topk_long_rows(int N_c, int k);
int topk_wmax_ld(int N_c);
size_t topk_wmax_bytes(long long rows, int N_c);

// ---- indexer ----
int indexer_group_tokens(int n_q);
int indexer_box_rows(int T);
// wmax non-null (decode groups, T = 1): the epilogue also writes, per row
// (b * n_q_rows + i of the chunk), the largest score key (score_key) of every
// 32 consecutive visible entries j to wmax[row * wmax_ld + j / 32].
// scores: fp32, or bf16 (nearest even) when score_bf16.
// head_w ([B, n_q, H_I] or null) and relu: the weighted / ReLU variant,
// s = sk * sum_h w_h sq_h max(<q_h, k>, 0).
// zero_words (n_zero words, or null): cleared by the kernel's first CTA for
// the kernel that follows (the fused route's top-k row counters).
cudaError_t launch_indexer_tc(bool fp8, int T, const CUtensorMap& tq, const CUtensorMap& tk,
                              const float* q_scale, const float* head_w, bool relu, const float* k_scale,
                              void* scores, bool score_bf16, int B,
                              int n_q_total, int i_start, int n_q_rows, QPos q_pos0, int m, int Nc,
                              int num_sms, uint32_t* wmax, int wmax_ld, bool kfp4, cudaStream_t s,
                              uint32_t* zero_words = nullptr, int n_zero = 0);
cudaError_t launch_indexer_f32(const float* q, const float* q_scale, const float* head_w, bool relu,
                               const float* k, const float* k_scale, void* scores, bool score_bf16, int B,
                               int n_q_total, int i_start, int n_q_rows,
                               QPos q_pos0, int m, int Nc, int HI, int dI, cudaStream_t s);
cudaError_t launch_fp4_to_e4m3(const uint8_t* packed, const uint8_t* sc, uint8_t* x8, float* S,
                               long long rows, int d, cudaStream_t s);

// ---- attention ----
template <typename TIO> struct AttnArgsT {
    const TIO* q;        // [B, n_q, H, D]
    const TIO* k_ptr;    // [B, N_kv, D]
    const TIO* v_ptr;    // [B, N_kv, D]
    TIO* out;            // [B, n_q, H, D]
    float* lse;          // [B, n_q, H] or null
    const int32_t* topk; // [B, n_q, k] (mode 0)
    float* part_o;       // [n_splits, B*n_q, H, D] when n_splits > 1
    float* part_ml;      // [n_splits, B*n_q, H, 2]
    long long q_pos0, window;
    float scale_log2;    // softmax scale * log2(e)
    int mode;            // 0 sparse, 1 closed blocks, 2 window
    int B, n_q, N_kv, k, m, n_splits;
    // KV heads: K / V are [B, N_kv, H_kv, D]; query head h (of H_tot) reads KV
    // head h / G, G = H_tot / H_kv.  (1, H_tot, H_tot) is one shared KV head.
    int H_kv = 1, H_tot = 0, G = 0;
};
bool attn_simt_supported(int H, int D);
// H: query heads per KV head (G); a.H_tot, a.H_kv, a.G describe the layout.
template <typename TIO>
cudaError_t launch_attn_simt(const AttnArgsT<TIO>& a, int H, int D, cudaStream_t s);
// merges split partials (a.part_o, a.part_ml) into a.out / a.lse
cudaError_t launch_attn_combine(const AttnArgsT<__nv_bfloat16>& a, int H, int D, cudaStream_t s);

// tcgen05 attention (BF16, D = 128, H in {64, 128}); tensor maps over
// Q [B*n_q*H, 128] (box attn_tc_q_box_rows rows) and K / V [B*N_kv, 128]
// (box 128 rows for the dense modes, 1 row for the sparse mode's gathers),
// 64-column boxes with 128-byte swizzle.
struct AttnTcParams {
    const int32_t* topk;   // [B, n_q, k] (mode 0)
    const __nv_bfloat16* k_rows;   // K [B * N_kv, 128] (mode 0: rows gathered with cp.async)
    const __nv_bfloat16* v_rows;   // V [B * N_kv, 128]
    __nv_bfloat16* out;    // [B, n_q, H, 128]
    float* lse;            // [B, n_q, H] or null
    float* part_o;         // [n_splits, B*n_q, H, 128] when n_splits > 1
    float* part_ml;        // [n_splits, B*n_q, H, 2]
    long long q_pos0, window;
    float scale_log2;      // softmax scale * log2(e)
    int B, n_q, N_kv, k, m, H;
    int T;                 // query tokens per CTA
    int n_splits, split_len;   // key-set slices of split_len (a multiple of 128)
};
bool attn_tc_supported(int H, int D);
int attn_tc_tokens_per_cta(int mode, int H);
int attn_tc_q_box_rows(int mode, int H);
cudaError_t launch_attn_tc(int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const AttnTcParams& p, cudaStream_t s);

}  // namespace csa
