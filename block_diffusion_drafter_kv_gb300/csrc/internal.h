// Internal interfaces between the kernels and the C ABI glue (not installed).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfl {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// ---------------------------------------------------------------- weight-streaming GEMM
// Y = X · Wᵀ over a weight matrix streamed once from HBM: the weight tile (128 output rows
// x 64 k) is the 128-row A operand of tcgen05.mma, the <= 256 activation rows are the N
// operand. Work is split "stream-K" style: the (tile, k-block) units are divided evenly
// over the CTAs; a tile split between CTAs is reduced in a fixed order by the CTA whose
// last tile it is, once the others' partials are in, so results never depend on timing.
enum GemvOp : int {
  OP_PLAIN = 0,   // Y fp32
  OP_FC = 1,      // context fusion: cfeat = bf16(F * g_ctx), per-tile sum of squares of F
  OP_KV = 2,      // injection: scale by 1/rms, RoPE on K, append K/V to the cache
  OP_QKV = 3,     // block q/k/v: scale by 1/rms, RoPE on q and k, q -> q_buf, k/v -> cache
  OP_RESID = 4,   // x += acc; xg = bf16(x * gain); per-tile sum of squares of x
  OP_SWIGLU = 5,  // act = bf16(silu(gate/rms) * up/rms)
  OP_LMHEAD = 6,  // z = acc/rms; optional logits; running argmax; last CTA writes drafts
};

constexpr int kMaxAMaps = 16;
constexpr int kPageRows = 64;      // positions per page of a paged KV cache (= attention key tile)
constexpr int kMaxCtas = 256;      // workspace partial slots are sized for this many CTAs
constexpr int kMaxPassRows = 256;  // activation rows per GEMM pass (MMA N <= 256 per plane)

struct GemvParams {
  CUtensorMap amap[kMaxAMaps];  // weight maps, box 64 (k) x 64 (rows), 128-byte swizzle
  CUtensorMap bmap;             // activation map, box 64 (k) x 16*NB rows [x 1 tap]
  int b_lo;                     // rows from a high-plane row to its low plane in bmap; 0: no low plane
  int n_amaps;
  int tile_start[kMaxAMaps + 1];  // map i covers tiles [tile_start[i], tile_start[i+1])
  int pair_mode;                  // rows 0-63 of tile t from map 0 row 64t, rows 64-127 from map 1 row 64t
  int T;                          // output tiles of 128 rows
  int KB;                         // k-blocks of 64 per tile
  int b3d;                        // B operand: 3-D map over [taps][rows][Ht]
  int b_kb_per_tap;               // Ht / 64 when b3d
  int b_row0;                     // row coordinate of the pass in the B operand
  int grow0;                      // global row id of local row 0 (positions, validity)
  int out_row0;                   // row of local row 0 in the output buffers
  int ss_row0;                    // row of local row 0 in ss_in
  int n_valid;                    // rows with global id < n_valid are real (draft ops)
  int op;
  int n_out;                      // valid output features (ragged vocab)
  // split-K reduction state (workspace)
  float* part;
  int* tile_cnt;
  int* cta_cnt;
  int* err;
  // RMSNorm folded into the epilogue: inv_rms[row] = rsqrt(sum_p ss_in[p*ss_stride + row] / H + eps)
  const float* ss_in;
  int ss_parts;
  int ss_stride;
  float* ss_out;  // [T][ss_stride]
  float eps;
  int H;
  const __nv_bfloat16* gain;
  // outputs
  float* y;                 // PLAIN: Y; RESID: residual x
  int y_ld;
  __nv_bfloat16* yb;        // FC: cfeat; RESID: xg; SWIGLU: act (bf16 high plane)
  int yb_ld;
  int yb_lo;                // rows from a yb row to its low plane; 0: write the high plane only
  __half* qh;               // QKV: post-RoPE queries, fp16, [rows][nq*d]
  float* trace;             // RESID: optional residual trace
  // RoPE and caches
  const float* rope_cos;    // [cap][d/2]
  const float* rope_sin;
  int d;
  __half* kc;               // K cache (post-RoPE), fp16: [L][max_batch][cap][nkv][d]
  __half* vc;               // V cache, fp16, same layout
  int nkv, cap, max_batch, layer;
  int layer_rows;           // rows (positions) per layer of the cache: max_batch * cap, or pages * kPageRows
  const int* page_table;    // paged cache: [max_batch][pages_per_seq] page ids, or null (sequence-major)
  int pages_per_seq;
  int* len;
  const int* n_new;
  int rows_per_seq;         // KV: row stride per sequence; draft ops: block size B
  int batch;
  int commit_len;
  // LM head
  float* logits;
  int vocab;
  float* best_v;            // [kMaxCtas][kMaxPassRows]
  int* best_i;
  int* drafted;             // drafts d_1..d_{B-1} of every sequence; with lm_all_rows, argmax of every row
  int lm_all_rows;          // the target's greedy tokens: every row's argmax, at its row index
};

// Up to kMaxPhases projections run back to back in one persistent launch: phase p+1 may
// read what phase p wrote (grid barrier in between); weights of phase p+1 are streamed
// before the barrier. Every CTA must be resident at once (grid <= SMs, one CTA per SM).
constexpr int kMaxPhases = 8;
struct GemvChain {
  GemvParams ph[kMaxPhases];
  int n_phases;
  int* bar;       // [kMaxPhases] arrival counters, zero at launch; cleared by the last CTA out
  int* exit_cnt;  // [1]
  unsigned long long* tl;  // per-CTA timeline records (kTlWords each) or null
  int tl_id;               // launch id written into the records
  unsigned long long wait_ns;  // limit of every wait in the kernel
  int bar_extra;           // added to every grid-barrier target: 0, or 1 in the timeout self-test
};

// Timeline record of one CTA (kTlWords 64-bit words, %globaltimer nanoseconds):
//   [0] (kind << 32) | launch id   [1] SM id   [2] entry   [3] set-up done
//   [4 + 4p] phase p: producer starts it   [5 + 4p] its input is ready (previous phase / kernel)
//   [6 + 4p] first operand stage landed    [7 + 4p] epilogue done with it   (p < 8)
//   [kTlExit] exit
constexpr int kTlWords = 37;
constexpr int kTlExit = kTlWords - 1;
enum TlKind : int { TL_GEMV = 1, TL_ATTN = 2, TL_EMBED = 3, TL_VERIFY = 4 };

// Kernel variant for nb activation row groups of 16 (1, 2, 4, 8 or 16); `pref` selects
// among the nb == 1 variants. KB of a launch counts k-stages of 64 * gemv_variant_ksub(v).
int gemv_variant(int nb, int pref);
int gemv_variant_ksub(int variant);
int gemv_variant_ksub1(int nb);  // the one-box-per-stage variant for nb
int launch_gemv(const GemvChain& p, int variant, int n_ctas, cudaStream_t stream, bool pdl);
int gemv_set_attributes();

// ---------------------------------------------------------------- block attention
struct AttnParams {
  CUtensorMap kmap;  // 3-D over this layer's fp16 K cache: {d, nkv, max_batch*cap}, box {64, 1, 64}
  CUtensorMap vmap;  // 3-D over this layer's fp16 V cache: box {64, 1, 64}
  CUtensorMap kmap32, vmap32;  // the same in boxes of 32 positions (tensor-core flat kernel)
  const __half* q;   // [rows][nq*d], row = s*B + i, post-RoPE, fp16
  __nv_bfloat16* o;  // [rows][nq*d] high plane; the low plane follows o_lo rows further on
  int o_lo;
  const int* len;
  int* err;
  int B, nq, nkv, d, cap;
  const int* page_table;   // paged cache: [max_batch][pages_per_seq] page ids (tile t of a sequence is its
  int pages_per_seq;       // page t), or null: sequence s's keys start at row s * cap
  int n_pages;             // pages in the pool (paged cache)
  float scale_log2;        // log2(e) / sqrt(d)
  unsigned long long* tl;  // timeline records (kTlWords per CTA) or null
  int tl_id;
  unsigned long long wait_ns;  // limit of every wait in the kernel
  int key_groups;          // 1, or 2 (GQA groups of at most 4 heads): warps taking alternate tiles
  // flat key split (attn_flat_kernel) only
  int batch;
  float* part;             // [2 * CTAs] slots of (group*16 rows x (d outputs), then (max, sum, 0, 0) per row)
  int* cnt;                // [batch][nkv] arrival counters, zero between launches
};
constexpr int kAttnFlatMaxBatch = 4096;  // sequences per flat-split launch (a shared-memory prefix table)
int launch_attention(const AttnParams& p, int batch, int split, cudaStream_t stream, bool pdl);
int launch_attention_flat(const AttnParams& p, int n_ctas, cudaStream_t stream, bool pdl);
// The flat split on the tcgen05 tensor cores (head dim 128, 4 query heads per KV head,
// B <= 16); attn_tc_supported says whether p qualifies.
bool attn_tc_supported(const AttnParams& p);
int launch_attention_flat_tc(const AttnParams& p, int n_ctas, cudaStream_t stream, bool pdl);
int attn_tc_set_attributes();
int attn_set_attributes();
int attn_resident_clusters(int split);

// ---------------------------------------------------------------- small kernels
struct EmbedParams {
  const __nv_bfloat16* embed;     // [V][H]
  const __nv_bfloat16* mask_emb;  // [H]
  const __nv_bfloat16* gain;      // g_attn of layer 0
  const int* last_token;
  const int* len;
  float* x;                       // [rows][H]
  __nv_bfloat16* xg;              // [rows][H] high plane; low plane xg_lo rows further on
  int xg_lo;
  float* ss;                      // [rows]
  float* trace;                   // [rows][H] or null
  int* err;
  int B, H, V, cap;
  unsigned long long* tl;
  int tl_id;
};
int launch_embed(const EmbedParams& p, int batch, cudaStream_t stream, bool pdl);

struct VerifyParams {
  const float* logits;  // [batch][B][V]
  const int* drafted;   // [batch][B-1]
  int* accept_len;
  int* committed;
  int* last_token;
  float* part_v;        // [batch][B][chunks]
  int* part_i;
  int* seq_cnt;         // [batch]
  int* err;
  int B, V, chunks, chunk_len;
  unsigned long long* tl;
  int tl_id;
};
int launch_verify(const VerifyParams& p, int batch, cudaStream_t stream, bool pdl);

// Sampling-mode verification (temperature > 0): speculative sampling with the drafts as
// point proposals. Same chunked grid as verify_kernel; the partials are per-chunk
// (max, sum of exp) of z / T.
struct VerifySampleParams {
  const float* logits;    // [batch][B][V]
  const int* drafted;     // [batch][B-1]
  const float* uniforms;  // [batch][B]: accept tests u_0..u_{B-2}, then w for the sampled token
  float inv_temp;
  int* accept_len;
  int* committed;
  int* last_token;
  float* part_m;          // [batch][B][chunks]
  float* part_s;
  int* seq_cnt;           // [batch]
  int* err;
  int B, V, chunks, chunk_len;
};
int launch_verify_sampling(const VerifySampleParams& p, int batch, cudaStream_t stream, bool pdl);

// Fused target-side verification: rows of the target's last hidden states -> the bf16
// planes of h * g (the LM head's operand) and each row's sum of squares; then, once the
// row argmaxes g are known, the longest-prefix acceptance.
struct TargetPrepParams {
  const __nv_bfloat16* hidden;  // [rows][Ht]
  const __nv_bfloat16* gain;    // [Ht]
  __nv_bfloat16* xg;            // [rows][Ht] high plane; low plane xg_lo rows further on
  int xg_lo;
  float* ss;                    // [rows]
  int Ht;
};
int launch_target_prep(const TargetPrepParams& p, int rows, cudaStream_t stream, bool pdl);

struct AcceptParams {
  const int* g;         // [batch][B] the target's greedy tokens
  const int* drafted;   // [batch][B-1]
  int* accept_len;
  int* committed;
  int* last_token;
  int batch, B;
};
int launch_accept(const AcceptParams& p, cudaStream_t stream, bool pdl);

int launch_plant(float* logits, const int* drafted, const uint8_t* masks, int n_steps, const int* step,
                 int batch, int B, int V, float bump, int* saved, cudaStream_t stream);
int launch_unplant(float* logits, int* step, int n_steps, int batch, int B, const int* saved,
                   cudaStream_t stream);

}  // namespace dfl
