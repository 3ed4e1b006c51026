/*
 * dflash.h — C ABI of the GB300 (sm_103a) DFlash draft-and-verify step.
 *
 * DFlash drafts a whole block of future tokens with a small block-diffusion drafter in
 * one forward pass; the target verifies the block in parallel and keeps the longest
 * valid prefix. The drafter is conditioned on the target: hidden states from several
 * target layers are fused into one compact target-context feature, which is injected
 * into the Key and Value projections of every draft layer, where it stays in the draft
 * KV cache across drafting iterations.
 *   - jansverre.net, "DFlash: slik kan spekulativ dekoding gi opptil 6x raskere
 *     AI-inferens", section "Hva gjør DFlash annerledes enn vanlig spekulativ dekoding?"
 *   - theaistack.guide, "DFlash Crea Blocchi Interi di Token Contemporaneamente ...",
 *     sections "Come funziona il drafting a blocchi" and "L'idea chiave: Il target sa
 *     meglio"
 *   - bpdata.com DFlash article (Hungarian), introduction and section "Hogyan működik a
 *     DFlash spekulatív dekódolás?"
 *
 * One step is three calls on one stream: dflash_inject_ctx -> dflash_draft_block ->
 * (target forward, outside this library) -> dflash_verify_greedy.
 *
 * Conventions for every call:
 *   - All device memory (weights, KV caches, per-sequence state, workspace, inputs and
 *     outputs) is allocated and owned by the caller. The library allocates no device
 *     memory at any point; it keeps only a host-side handle.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream) and return a status code. Errors that the host can see (null
 *     pointers, sizes out of range, unsupported shapes) return before any launch.
 *   - Per-sequence lengths and token ids live on the device, so a step never needs a
 *     host synchronisation and can be captured in a CUDA graph. Errors found by a kernel
 *     (a capacity overflow, a token id out of range, a bounded wait that gave up) set a
 *     flag in the workspace; kernels then skip the offending writes. Read and clear it
 *     with dflash_read_device_error().
 *   - bf16 means IEEE bfloat16 stored as 16-bit words; all matrices are row-major.
 *   - Device pointers handed to the library must be 16-byte aligned; weight and
 *     activation row strides are multiples of 16 bytes by construction of the shapes
 *     dflash_create accepts.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ------------------------------------------------ */
#define DFLASH_OK 0
#define DFLASH_E_INVAL (-1)    /* bad argument: null pointer, size out of range, misalignment */
#define DFLASH_E_CONFIG (-2)   /* drafter shape not supported by these kernels */
#define DFLASH_E_CAPACITY (-3) /* batch/block/rows beyond what the config or workspace holds */
#define DFLASH_E_CUDA (-4)     /* a CUDA runtime or driver call failed */
#define DFLASH_E_STATE (-5)    /* dflash_bind_state has not been called */

/* ---- device error flag bits (dflash_read_device_error) ---------------------------- */
#define DFLASH_DEV_TIMEOUT 1   /* a bounded wait inside a kernel gave up; its results are void */
#define DFLASH_DEV_CAPACITY 2  /* a write past a sequence's KV capacity was skipped */
#define DFLASH_DEV_TOKEN 4     /* a token id outside [0, vocab) was seen; the row was skipped */

/* ---- drafter shape ---------------------------------------------------------------- */
typedef struct dflash_config {
  int32_t hidden;        /* H: drafter hidden size, multiple of 128, at most 8192 */
  int32_t n_heads;       /* nq: query heads */
  int32_t n_kv_heads;    /* nkv: key/value heads; nq % nkv == 0, nq/nkv <= 8 */
  int32_t head_dim;      /* d: 64 or 128; nq*d and nkv*d multiples of 128 */
  int32_t n_layers;      /* L: draft layers, 1..16 */
  int32_t intermediate;  /* I: SwiGLU inner size, multiple of 64 */
  int32_t vocab;         /* V: vocabulary size, >= 2 */
  int32_t n_taps;        /* k: tapped target layers, 1..16 */
  int32_t target_hidden; /* Ht: target hidden size, multiple of 64 */
  float rope_theta;      /* RoPE base */
  float rms_eps;         /* RMSNorm epsilon */
  int32_t max_block;     /* largest block B accepted by draft/verify, 1..16 */
  int32_t max_batch;     /* largest number of sequences per call, 1..256 */
  int32_t kv_capacity;   /* positions per sequence in the KV cache */
} dflash_config;

/* ---- weights (device pointers, bf16, caller-owned, registered once) --------------- */
typedef struct dflash_layer_weights {
  const void* wq;     /* [nq*d, H]  query projection */
  const void* wk;     /* [nkv*d, H] key projection; also projects the injected context */
  const void* wv;     /* [nkv*d, H] value projection; also projects the injected context */
  const void* wo;     /* [H, nq*d]  attention output projection */
  const void* w_gate; /* [I, H]     SwiGLU gate */
  const void* w_up;   /* [I, H]     SwiGLU up */
  const void* w_down; /* [H, I]     SwiGLU down */
  const void* g_attn; /* [H]        RMSNorm gain before attention */
  const void* g_mlp;  /* [H]        RMSNorm gain before the MLP */
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* w_fc;     /* [H, k*Ht] fusion of the k concatenated target hidden states */
  const void* g_ctx;    /* [H]       RMSNorm gain of the fused context feature */
  const void* embed;    /* [V, H]    token embedding (slot 0 of a block) */
  const void* mask_emb; /* [H]       mask embedding (slots 1..B-1 of a block) */
  const void* g_final;  /* [H]       final RMSNorm gain */
  const void* lm_head;  /* [V, H]    LM head */
  const dflash_layer_weights* layers; /* host array of n_layers entries */
} dflash_weights;

typedef struct dflash_handle dflash_handle;

/* Validate a shape without touching the GPU. Returns DFLASH_OK or DFLASH_E_CONFIG. */
int dflash_config_check(const dflash_config* cfg);

/* Workspace bytes dflash_bind_state needs for this shape (0 if the shape is invalid).
 * The workspace holds activations, split-K partials, reduction counters, the RoPE
 * tables and the device error flag. */
size_t dflash_workspace_size(const dflash_config* cfg);

/* Register a drafter. Copies the config, records the weight pointers (which must stay
 * valid until dflash_destroy) and encodes their TMA descriptors on the host. Uses the
 * current CUDA device. *out receives the handle. */
int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out);

/* Release the host handle. Device memory stays the caller's. */
int dflash_destroy(dflash_handle* h);

/* Bind caller-owned state:
 *   k_cache           fp16 [L][max_batch][kv_capacity][nkv][d], K after RoPE.
 *   v_cache           fp16 [L][max_batch][kv_capacity][nkv][d].
 *                     IEEE half precision: 11 significant bits (the attention scores are
 *                     the step's most rounding-sensitive quantity, and the value products
 *                     follow them), 2 bytes per element; values beyond +-65504 overflow, so
 *                     the drafter's K and V must stay within that range.
 *                     Both zero-initialised by the caller. Positions [len, len+B) are used
 *                     as scratch for the block's own keys/values during a draft.
 *   len               int32 [max_batch] injected positions per sequence (device)
 *   last_token        int32 [max_batch] slot-0 token of the next block (device)
 *   workspace         dflash_workspace_size(cfg) bytes, 256-byte aligned
 * Fills the RoPE tables and clears the workspace (synchronous; call once before use). */
int dflash_bind_state(dflash_handle* h, void* k_cache, void* v_cache, int32_t* len,
                      int32_t* last_token, void* workspace, size_t workspace_bytes);

/* Bind caller-owned state with a paged KV cache, for many ragged sequences sharing one pool:
 *   k_pool, v_pool    fp16 [L][n_pages * 64][nkv][d]: pages of 64 positions
 *   page_table        int32 [max_batch][pages_per_seq] on the device: sequence s keeps
 *                     position p at row page_table[s][p / 64] * 64 + p % 64 of every layer.
 *                     Read by the kernels at every call: the caller may hand out new pages
 *                     between calls (the pages a sequence uses must not be shared).
 *                     pages_per_seq * 64 >= kv_capacity; page ids in [0, n_pages) (others set
 *                     DFLASH_DEV_CAPACITY and the affected rows are skipped).
 *   len, last_token, workspace: as for dflash_bind_state.
 * Every other call behaves as with dflash_bind_state; results are bit-identical. */
int dflash_bind_state_paged(dflash_handle* h, void* k_pool, void* v_pool, int32_t n_pages,
                            const int32_t* page_table, int32_t pages_per_seq, int32_t* len,
                            int32_t* last_token, void* workspace, size_t workspace_bytes);

/* KV injection (theaistack.guide, "L'idea chiave: Il target sa meglio"): for every new
 * position, concatenate the k tapped target hidden states (tap order), fuse them with
 * w_fc, RMSNorm with g_ctx into the context feature c, project c with every layer's
 * Wk and Wv, apply RoPE to the keys at their absolute positions and append K/V to the
 * cache at len[s] + r; then len[s] += n_new[s].
 *   hidden        bf16 [k][batch * rows_per_seq][Ht]; sequence s's new rows are rows
 *                 s*rows_per_seq + r for r < n_new[s]
 *   rows_per_seq  row stride between sequences in `hidden` (host int, >= 1)
 *   n_new         int32 [batch] on the device, 0 <= n_new[s] <= rows_per_seq
 * Rows past n_new[s] are read but never written anywhere. A sequence that would pass
 * kv_capacity sets DFLASH_DEV_CAPACITY and its overflowing rows are skipped. The
 * result for a row depends only on that row, so two incremental injections give
 * bit-identical caches to one injection of the same positions. */
int dflash_inject_ctx(dflash_handle* h, const void* hidden, int32_t rows_per_seq,
                      const int32_t* n_new, int32_t batch, void* stream);

/* One block-diffusion draft pass (jansverre.net, "Hva gjør DFlash annerledes enn vanlig
 * spekulativ dekoding?": the whole masked block is denoised in a single forward pass).
 * Slot 0 of sequence s embeds last_token[s]; slots 1..B-1 hold the mask embedding;
 * slot i sits at position len[s] + i. Each layer: RMSNorm, Q/K/V projection with RoPE,
 * bidirectional attention over the injected context [0, len[s]) and the block's own B
 * keys, output projection, RMSNorm, SwiGLU MLP (pre-norm, residual adds); then the final
 * RMSNorm, the LM head on slots 1..B-1 and argmax (lowest index on ties).
 *   drafted   int32 [batch][B-1] out: d_1..d_{B-1}
 *   logits    fp32 [batch][B-1][V] out, or NULL (parity checks only; costs bandwidth);
 *             16-byte aligned
 *   x_trace   fp32 [L+1][batch*B][H] out, or NULL: block input then the residual after
 *             every layer (parity checks only); 16-byte aligned
 * A misaligned logits or x_trace returns DFLASH_E_INVAL before any launch.
 * Needs len[s] + B <= kv_capacity (else DFLASH_DEV_CAPACITY and the sequence's cache
 * writes are skipped). len is not changed. */
int dflash_draft_block(dflash_handle* h, int32_t batch, int32_t block, int32_t* drafted,
                       float* logits, float* x_trace, void* stream);

/* Greedy verification (bpdata.com DFlash article, introduction: the target accepts the
 * longest valid prefix): g_i = argmax target_logits[s][i] (lowest index on ties);
 * j = the number of leading i with drafted[s][i] == g_i (i < B-1); tau = j + 1.
 *   target_logits  fp32 [batch][B][V], finite, 16-byte aligned
 *   drafted        int32 [batch][B-1]
 *   accept_len     int32 [batch] out: tau in [1, B]
 *   committed      int32 [batch][B] out: g_0..g_{tau-1}, then -1
 * Also writes last_token[s] = g_{tau-1} (the next block's slot 0). Committed tokens are
 * always the target's own greedy tokens, so the output equals target-only greedy
 * decoding. The caller injects the tau accepted positions on the next step. */
int dflash_verify_greedy(dflash_handle* h, const float* target_logits, const int32_t* drafted,
                         int32_t batch, int32_t block, int32_t* accept_len, int32_t* committed,
                         void* stream);

/* Verification when the target samples at a temperature (7minutos.es, "Casos de uso con
 * ejemplos": the method is also measured under sampling). The pages state no accept rule;
 * this is standard speculative sampling with the drafter's argmax as a point proposal,
 * which keeps the committed tokens distributed as the target's own samples:
 *   p_i = softmax(target_logits[s][i] / temperature)
 *   accept d_{i+1} (= drafted[s][i]) while u_i < p_i(d_{i+1}), i = 0..B-2;
 *   at the first rejection (row j) the last token is sampled from p_j without d_{j+1},
 *   renormalised; with every draft accepted it is the bonus token sampled from p_{B-1}.
 *   The token is the first index whose cumulative probability exceeds w (inverse CDF).
 *   target_logits  fp32 [batch][B][V], finite
 *   drafted        int32 [batch][B-1]
 *   uniforms       fp32 [batch][B] in [0, 1): u_0..u_{B-2}, then w (the caller's random
 *                  numbers; the library draws none)
 *   temperature    > 0
 *   accept_len     int32 [batch] out: tau in [1, B] (accepted drafts plus the sampled token)
 *   committed      int32 [batch][B] out: d_1..d_{tau-1}, the sampled token, then -1
 * Writes last_token[s] = the sampled token. Sums run in fp32: where a uniform lies within
 * about 1e-6 of a decision boundary the outcome may differ from an exact evaluation. */
int dflash_verify_sampling(dflash_handle* h, const float* target_logits, const int32_t* drafted,
                           const float* uniforms, float temperature, int32_t batch, int32_t block,
                           int32_t* accept_len, int32_t* committed, void* stream);

/* Greedy verification starting from the target's last hidden states (bpdata.com DFlash
 * article, introduction: the target checks the whole drafted block in one parallel pass and
 * keeps the longest valid prefix). Fuses the target's own final RMSNorm (gain target_gain,
 * the drafter's rms_eps), its LM head and the argmax of every block position into the
 * library's weight-streaming kernels, then applies the acceptance rule of
 * dflash_verify_greedy, so the [batch][B][V] fp32 logits never exist.
 *   target_hidden   bf16 [batch * B][Ht] (Ht = target_hidden of the config, <= 8192):
 *                   the target's last-layer hidden state at each block position
 *   target_gain     bf16 [Ht] the target's final RMSNorm gain
 *   target_lm_head  bf16 [V][Ht] the target's LM head (V = vocab of the config)
 *   drafted, accept_len, committed: as for dflash_verify_greedy; last_token[s] is written.
 * Pointers 16-byte aligned (token arrays 4-byte); ties go to the lowest index. */
int dflash_verify_greedy_hidden(dflash_handle* h, const void* target_hidden, const void* target_gain,
                                const void* target_lm_head, const int32_t* drafted, int32_t batch, int32_t block,
                                int32_t* accept_len, int32_t* committed, void* stream);

/* Weight-streaming bf16 GEMM of the draft path, exposed for testing the engine alone:
 * Y[r][m] = sum_k X[r][k] * W[m][k] in fp32 accumulation.
 *   W  bf16 [n_out][K] (K multiple of 64), X bf16 [rows][K] (any rows; passes of 256),
 *   Y  fp32 [rows][n_out] out. Uses the handle's bound workspace for split-K partials. */
int dflash_linear_bf16(dflash_handle* h, const void* W, int32_t n_out, int32_t K, const void* X,
                       int32_t rows, float* Y, void* stream);

/* Copy the device error flag to *flags once the work queued on `stream` so far has
 * finished (it waits for that stream only, not for the whole device). With `clear`
 * non-zero it then zeroes the flag and every arrival counter in the workspace, which a
 * kernel that gave up a bounded wait may have left part-counted; the handle is then
 * usable again. Work of this handle must not be in flight on other streams meanwhile. */
int dflash_read_device_error(dflash_handle* h, int32_t* flags, int32_t clear, void* stream);

/* Per-handle settings (not part of the method; defaults suit GB300):
 *   DFLASH_OPT_WAIT_LIMIT_NS  limit of every spin-wait inside a kernel (mbarriers, grid
 *                             barriers, cluster peers), in ns, 1e5..6e10; default 2e9.
 *                             Past it the kernel sets DFLASH_DEV_TIMEOUT and returns.
 *   DFLASH_OPT_CHAIN_MAX      projections per persistent launch, 1..8; default 8
 *   DFLASH_OPT_GEMV_VARIANT   weight-streaming variant of single-row-group passes, 0..5;
 *                             default 3 (4 k-boxes per stage, 2 stages)
 *   DFLASH_OPT_ATTN_SPLIT     CTAs per attention cluster, 0..16; 0 (default) chooses from
 *                             the SM count
 *   DFLASH_OPT_ATTN_KEY_GROUPS  warps per query head in the attention kernel, 1..2; with 2
 *                             (default; GQA groups of at most 4 heads) the two take
 *                             alternate key tiles and are combined after the key loop
 *   DFLASH_OPT_INJECT_PASS_ROWS  rows per injection pass: 16, 32, 64, 128 or 256; default 16 x
 *                             the row groups of max_batch * max_block (at most 256). Every pass
 *                             streams the fusion and K/V weights once, so wide passes make
 *                             long prefills cheaper and short injections dearer. Injections
 *                             at one width give bit-identical K/V however positions are
 *                             chunked into calls; different widths may differ in the last
 *                             bits (within the parity tolerance), so set it before the first
 *                             injection and keep it.
 *   DFLASH_OPT_ATTN_MODE      attention kernel: 0 (default) a cluster of 12 CTAs per (sequence,
 *                             KV head) splitting its keys where every pair gets one at once,
 *                             otherwise one flat list of every pair's key tiles split evenly
 *                             over the SMs (several, ragged or long contexts): on the tcgen05
 *                             tensor cores (head dim 128, 4 query heads per KV head, an even
 *                             KV head count, at most 1024 sequences) where batch x KV heads is
 *                             at most the SM count, else on the mma.sync path; 1 always
 *                             clusters; 2 always the flat split, on the tensor cores where the
 *                             shape allows (at most 4096 sequences); 3 the flat split on the
 *                             mma.sync path
 * Values out of range return DFLASH_E_INVAL and leave the setting unchanged. */
#define DFLASH_OPT_WAIT_LIMIT_NS 1
#define DFLASH_OPT_CHAIN_MAX 2
#define DFLASH_OPT_GEMV_VARIANT 3
#define DFLASH_OPT_ATTN_SPLIT 4
#define DFLASH_OPT_ATTN_KEY_GROUPS 5
#define DFLASH_OPT_INJECT_PASS_ROWS 6
#define DFLASH_OPT_ATTN_MODE 7
int dflash_set_option(dflash_handle* h, int32_t option, int64_t value);
int dflash_get_option(const dflash_handle* h, int32_t option, int64_t* value);

/* Self-test of the bounded waits (not part of the method): launches one chained
 * projection kernel (two plain projections through layer 0's output projection, writing
 * only the draft's residual scratch) whose second phase waits for a grid-barrier count
 * that no CTA reaches. Every waiting thread gives up after the handle's wait limit, the
 * kernel sets DFLASH_DEV_TIMEOUT, waits (bounded) for its copies and MMAs in flight,
 * releases its tensor memory and returns. Read and clear the flag with
 * dflash_read_device_error(clear = 1) before the next call. Use a short wait limit. */
int dflash_selftest_timeout(dflash_handle* h, void* stream);

/* Number of kernel launches the last call on this handle made. */
int32_t dflash_last_launch_count(const dflash_handle* h);

/* Per-launch tracing. `events` holds n_events caller-created cudaEvent_t handles (as void*;
 * n_events = 0 turns tracing off). While on, every call records events[0] on its stream
 * before its first launch and events[i] right after its i-th launch (while i < n_events),
 * so consecutive events bracket one kernel each. Launches are then fully serialised (no
 * programmatic overlap), which makes the traced durations conservative. The events must
 * outlive their use; the library does not own them. */
int dflash_trace_events(dflash_handle* h, void* const* events, int32_t n_events);

/* Per-CTA timeline. `records` is a caller-owned device buffer of n_records records of 37
 * uint64 words (n_records = 0 turns it off). While on, every CTA of every later launch
 * fills one record with %globaltimer nanosecond stamps, until the buffer is full:
 *   [0] (kind << 32) | launch number (kind 1 chained projection/attention kernel,
 *       2 standalone attention, 3 block embedding, 4 verification)   [1] SM id
 *   [2] entry   [3] set-up done
 *   [4+4p] phase p started   [5+4p] its input ready   [6+4p] first operand landed
 *   [7+4p] phase p finished (p < 8; other kernels fill [5] and a few of [6..9] only;
 *   the tensor-core flat attention kernel also [10] ns its producer waited for a free
 *   stage, [11] ns its MMA issuer had nothing to issue, [12] and [13] ns its softmax rows
 *   waited for scores and for the previous PV, [14] its key steps)
 *   [36] exit
 * Unset stamps keep whatever the buffer held, so clear it first. Calling this again
 * restarts at record 0. Stamps cost a few instructions per CTA. */
int dflash_timeline(dflash_handle* h, void* records, int64_t n_records);

/* Records filled since the last dflash_timeline call. */
int64_t dflash_timeline_used(const dflash_handle* h);

/* Human-readable text of a status code. */
const char* dflash_status_string(int status);

/* ---- greedy verification without any allocation -----------------------------------
 * The DFlash pages have no counterpart for this entry point; it exists for callers that
 * cannot allocate device memory at all, so cannot provide the workspace that
 * dflash_verify_greedy reads through a bound handle. Typical cases: code running inside
 * another inference engine whose memory pool forbids new allocations during decoding,
 * or a process that is only handed the logits and token buffers.
 *
 * Same result as dflash_verify_greedy (g_i = row argmax with the lowest index on ties;
 * tau = 1 + number of leading drafts equal to g_i; committed = g_0..g_{tau-1}, then -1)
 * and last_token[s] = g_{tau-1} is written to the caller's array. No handle is needed.
 * Its scratch (argmax partials and arrival counters, about 257 KB) is one fixed array
 * inside the library, which every GPU that loads the library keeps until the process
 * exits. Limits: batch <= DFLASH_NOALLOC_MAX_BATCH, block <= 16 (larger sizes return
 * DFLASH_E_CAPACITY before anything is launched) and 2 <= vocab <= DFLASH_NOALLOC_MAX_VOCAB
 * (DFLASH_E_INVAL otherwise). target_logits must be 16-byte aligned and the token
 * arrays 4-byte aligned (DFLASH_E_INVAL otherwise). It allocates no memory and calls no
 * allocating routine.
 *   - The first call on each device looks up the array's device address (a host-side
 *     symbol lookup). With lazy module loading (CUDA_MODULE_LOADING=LAZY) that lookup can
 *     load the library's device code on that device, which allocates the array and the
 *     code image. Make that first call before the region in which the caller may not
 *     allocate, and before any stream capture.
 *   - All calls share the one array. Calls whose work overlaps on the GPU (different
 *     streams without ordering, or different host threads) race and give wrong results;
 *     order them on one stream. Each call clears the counters it needs, so the
 *     contents left by an earlier call do not matter. */
#define DFLASH_NOALLOC_MAX_BATCH 64
#define DFLASH_NOALLOC_MAX_CHUNKS 32
#define DFLASH_NOALLOC_MAX_VOCAB (1 << 28)
int dflash_verify_greedy_noalloc(const float* target_logits, const int32_t* drafted, int32_t batch,
                                 int32_t block, int32_t vocab, int32_t* accept_len, int32_t* committed,
                                 int32_t* last_token, void* stream);

/* ---- synthetic target (benchmark harness, not part of DFlash) ---------------------
 * Stand-in for a target model inside a timed, graph-captured step: planting raises the
 * logit of drafted token d_{i+1} in row i by `bump` where plant_masks[step][s][i] != 0
 * (the target agrees with the draft there); unplanting restores the saved logits and
 * advances the device step counter (modulo n_steps).
 *   logits [batch][B][V] fp32, drafted [batch][B-1], plant_masks uint8 [n_steps][batch][B],
 *   step_counter int32 [1], saved: 2*batch*B int32 words of scratch. */
int dflash_synth_plant(float* logits, const int32_t* drafted, const uint8_t* plant_masks,
                       int32_t n_steps, const int32_t* step_counter, int32_t batch, int32_t block,
                       int32_t vocab, float bump, int32_t* saved, void* stream);
int dflash_synth_unplant(float* logits, int32_t* step_counter, int32_t n_steps, int32_t batch,
                         int32_t block, const int32_t* saved, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
