// C ABI of the DFlash draft-and-verify step (declared in include/dflash.h).
//
// Host side only: argument checks, the workspace layout, TMA descriptor encoding and the
// launch sequence of each call. Every step of the computation runs in the kernels of
// gemv.cu, attention.cu and small.cu.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "dflash.h"
#include "internal.h"

using namespace dfl;

namespace {

constexpr int kMaxChunks = 64;   // verification chunks per row
constexpr int kChainSlots = 64;  // barrier-counter sets, used round robin by consecutive launches
constexpr int kMaxLayersPerKvLaunch = kMaxAMaps / 2;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

struct WsLayout {
  size_t err, tile_cnt, cta_cnt, seq_cnt, rope_cos, rope_sin, part, best_v, best_i;
  size_t ss_fc, ss_x, ss_emb, cfeat, x, xg, q, o, act, vpart_v, vpart_i, chain_bar;
  size_t tgt_xg, tgt_ss, tgt_g;  // fused target-side verification
  size_t attn_part, attn_cnt;    // flat key-split attention: partial slots, per-pair counters
  size_t total;
  int R;          // draft rows allocated (multiple of 16)
  int max_tiles;  // tile counters
};

int max_tiles(const dflash_config& c) {
  const int d = c.head_dim;
  int t = ceil_div(c.vocab, 128);
  t = std::max(t, c.hidden / 128);
  t = std::max(t, (c.n_heads + 2 * c.n_kv_heads) * d / 128);
  t = std::max(t, c.intermediate / 64);
  t = std::max(t, 2 * kMaxLayersPerKvLaunch * c.n_kv_heads * d / 128);
  return t;
}

WsLayout layout_of(const dflash_config& c) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1), 256);
    return o;
  };
  const size_t H = c.hidden, d = c.head_dim, nq = c.n_heads, I = c.intermediate;
  L.R = static_cast<int>(align_up(static_cast<size_t>(c.max_batch) * c.max_block, 16));
  L.max_tiles = max_tiles(c);
  const size_t R = L.R;
  L.err = take(256);
  L.tile_cnt = take(static_cast<size_t>(L.max_tiles) * 4);
  L.cta_cnt = take(256);
  L.seq_cnt = take(static_cast<size_t>(c.max_batch) * 4);
  L.rope_cos = take(static_cast<size_t>(c.kv_capacity) * (d / 2) * 4);
  L.rope_sin = take(static_cast<size_t>(c.kv_capacity) * (d / 2) * 4);
  L.part = take(static_cast<size_t>(2) * kMaxCtas * kMaxPassRows * 128 * 4);
  L.best_v = take(static_cast<size_t>(kMaxCtas) * kMaxPassRows * 4);
  L.best_i = take(static_cast<size_t>(kMaxCtas) * kMaxPassRows * 4);
  L.ss_fc = take((H / 128) * kMaxPassRows * 4);
  L.ss_x = take((H / 128) * R * 4);
  L.ss_emb = take(R * 4);
  // bf16 activation operands hold a high plane of R rows and then the low plane (x - hi)
  L.cfeat = take(static_cast<size_t>(2 * kMaxPassRows) * H * 2);
  L.x = take(R * H * 4);
  L.xg = take(2 * R * H * 2);
  L.q = take(R * nq * d * 2);
  L.o = take(2 * R * nq * d * 2);
  L.act = take(2 * R * I * 2);
  L.vpart_v = take(static_cast<size_t>(c.max_batch) * c.max_block * kMaxChunks * 4);
  L.vpart_i = take(static_cast<size_t>(c.max_batch) * c.max_block * kMaxChunks * 4);
  L.chain_bar = take(static_cast<size_t>(kChainSlots) * (kMaxPhases + 4) * 4);
  L.tgt_xg = take(2 * R * static_cast<size_t>(c.target_hidden) * 2);
  L.tgt_ss = take(R * 4);
  L.tgt_g = take(R * 4);
  // flat attention slots: a head's 16 slots x its query heads, or two KV heads' (tensor-core kernel)
  L.attn_part = take(static_cast<size_t>(2) * kMaxCtas * 2 * (nq / c.n_kv_heads) * 16 * (d + 4) * 4);
  L.attn_cnt = take(static_cast<size_t>(c.max_batch) * c.n_kv_heads * 4);
  L.total = off;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool get_encoder() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// bf16 row-major [rows][inner], box 64 (inner) x box_rows, 128-byte swizzle.
bool enc2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [taps][rows][Ht], box 64 x box_rows x 1.
bool enc3d_hidden(CUtensorMap* m, const void* base, uint64_t Ht, uint64_t rows, uint64_t taps, uint32_t box_rows) {
  cuuint64_t dims[3] = {Ht, rows, taps};
  cuuint64_t strides[2] = {Ht * 2, Ht * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One layer's fp16 K or V cache [rows = max_batch*cap][nkv][d], box 64 (d, 128 bytes) x 1 head
// x 64 keys.
bool enc3d_cache(CUtensorMap* m, const void* base, uint64_t d, uint64_t nkv, uint64_t rows, uint32_t box_rows = 64) {
  cuuint64_t dims[3] = {d, nkv, rows};
  cuuint64_t strides[2] = {d * 2, nkv * d * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int nb_index(int nb) { return nb == 1 ? 0 : nb == 2 ? 1 : nb == 4 ? 2 : nb == 8 ? 3 : 4; }
int nb_for_rows(int rows) {
  int nb = 1;
  while (nb * 16 < rows && nb * 16 < kMaxPassRows) nb *= 2;
  return nb;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

}  // namespace

struct dflash_handle {
  dflash_config cfg{};
  dflash_weights w{};
  std::vector<dflash_layer_weights> layers;
  int device = 0;
  int n_sms = 0;
  // Rows per injection pass, fixed per handle (16 x the row groups of max_batch*max_block,
  // at most 128): every injection then uses the same kernel variant and split of the
  // weight, so a position's K/V are bit-identical however the positions are chunked.
  int inject_pass_rows = 16;
  int gemv_pref = 3;  // weight-streaming kernel variant for single-row-group launches
  int chain_slot = 0;
  int chain_max = kMaxPhases;  // projections per persistent launch (1 = one launch per projection)
  int attn_split = 0;          // CTAs per attention cluster (0: from the SM count)
  unsigned long long wait_ns = kDefaultWaitLimitNs;  // limit of every wait inside a kernel
  int attn_wide = 0;           // clusters of 12 the device holds at once (0: none)
  int attn_key_groups = 2;     // warps per query head in the attention kernel (taking alternate tiles)
  int attn_mode = 0;           // 0: clusters of 12 where they fit, else the flat key split; 1: clusters;
                               // 2: flat (tensor cores where the shape allows); 3: flat on mma.sync
  // weight descriptors
  CUtensorMap m_fc{}, m_lm{};
  std::vector<CUtensorMap> m_wq, m_wk, m_wv, m_wo, m_wg, m_wu, m_wd;
  // bound state
  bool bound = false;
  __half* kc = nullptr;
  __half* vc = nullptr;
  int layer_rows = 0;              // positions per layer of the cache
  const int* page_table = nullptr; // paged cache: [max_batch][pages_per_seq], or null
  int pages_per_seq = 0;
  int* len = nullptr;
  int* last_token = nullptr;
  uint8_t* ws = nullptr;
  WsLayout L{};
  CUtensorMap m_xg[5]{}, m_cfeat[5]{}, m_act[5]{}, m_o[5]{};  // by nb_index, over both planes
  CUtensorMap m_txg[5]{};  // the target's normed-hidden operand (fused verification), by nb_index
  std::vector<CUtensorMap> m_kcache, m_vcache;
  std::vector<CUtensorMap> m_kcache32, m_vcache32;  // the same caches in boxes of 32 positions
  int last_launches = 0;
  std::vector<cudaEvent_t> trace_ev;  // caller-owned events recorded around launches, or empty
  unsigned long long* tl_buf = nullptr;  // caller-owned timeline buffer, or null
  long long tl_cap = 0, tl_next = 0;     // records
  int tl_launch = 0;

  template <typename T>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
};

namespace {

void gemv_common(const dflash_handle* h, GemvParams& P) {
  P.part = h->at<float>(h->L.part);
  P.tile_cnt = h->at<int>(h->L.tile_cnt);
  P.cta_cnt = h->at<int>(h->L.cta_cnt);
  P.err = h->at<int>(h->L.err);
  P.eps = h->cfg.rms_eps;
  P.H = h->cfg.hidden;
  P.n_valid = 0x7fffffff;
  P.n_out = 0x7fffffff;
}

// Timeline records for a launch of n CTAs (null when the timeline is off or full).
unsigned long long* tl_take(dflash_handle* h, long long n) {
  if (!h->tl_buf || h->tl_next + n > h->tl_cap) return nullptr;
  unsigned long long* p = h->tl_buf + h->tl_next * kTlWords;
  h->tl_next += n;
  return p;
}

// Start of a call: reset the launch count; with tracing on, record event 0.
void call_begin(dflash_handle* h, cudaStream_t st) {
  h->last_launches = 0;
  if (!h->trace_ev.empty()) cudaEventRecord(h->trace_ev[0], st);
}

// After each launch: count it; with tracing on, record the event that closes it.
void note_launch(dflash_handle* h, cudaStream_t st) {
  ++h->last_launches;
  if (h->last_launches < static_cast<int>(h->trace_ev.size())) cudaEventRecord(h->trace_ev[h->last_launches], st);
}

// One persistent launch over a chain of projection phases (all with nb row groups). Each
// phase's KB arrives in 64-wide k-blocks; the kernel variant may stage several per step.
#define DFL_TRY(x)                \
  do {                            \
    const int _r = (x);           \
    if (_r != DFLASH_OK) return _r; \
  } while (0)

int run_chain_one(dflash_handle* h, const GemvParams* phases, int n, int nb, cudaStream_t st);

int run_chain(dflash_handle* h, const GemvParams* phases, int n, int nb, cudaStream_t st) {
  for (int p0 = 0; p0 < n; p0 += h->chain_max) DFL_TRY(run_chain_one(h, phases + p0, std::min(h->chain_max, n - p0), nb, st));
  return DFLASH_OK;
}

int run_chain_one(dflash_handle* h, const GemvParams* phases, int n, int nb, cudaStream_t st) {
  GemvChain C{};
  int v = gemv_variant(nb, h->gemv_pref);
  int ks = gemv_variant_ksub(v);
  for (int p = 0; p < n; ++p)
    if (phases[p].KB % ks != 0) {
      v = gemv_variant_ksub1(nb);
      ks = gemv_variant_ksub(v);
    }
  for (int p = 0; p < n; ++p) {
    C.ph[p] = phases[p];
    C.ph[p].KB /= ks;
  }
  C.n_phases = n;
  const int slot = h->chain_slot;
  h->chain_slot = (h->chain_slot + 1) % kChainSlots;
  C.bar = h->at<int>(h->L.chain_bar) + slot * (kMaxPhases + 4);
  C.exit_cnt = C.bar + kMaxPhases;
  const int G = std::min(h->n_sms, kMaxCtas);
  C.tl = tl_take(h, G);
  C.tl_id = h->tl_launch++;
  C.wait_ns = h->wait_ns;
  const int e = launch_gemv(C, v, G, st, h->trace_ev.empty());
  note_launch(h, st);
  return e == 0 ? DFLASH_OK : DFLASH_E_CUDA;
}

int run_gemv(dflash_handle* h, const GemvParams& P, int nb, cudaStream_t st) { return run_chain(h, &P, 1, nb, st); }


}  // namespace

extern "C" {

int dflash_config_check(const dflash_config* c) {
  if (!c) return DFLASH_E_INVAL;
  const int d = c->head_dim;
  bool ok = c->hidden >= 128 && c->hidden % 128 == 0 && c->hidden <= 8192 && c->n_heads >= 1 && c->n_kv_heads >= 1 &&
            c->n_heads % c->n_kv_heads == 0 && c->n_heads / c->n_kv_heads <= 8 && (d == 64 || d == 128) &&
            (c->n_heads * d) % 128 == 0 && (c->n_kv_heads * d) % 128 == 0 && c->n_layers >= 1 &&
            c->n_layers <= 16 && c->intermediate >= 64 && c->intermediate % 64 == 0 && c->vocab >= 2 &&
            c->n_taps >= 1 && c->n_taps <= 16 && c->target_hidden >= 64 && c->target_hidden % 64 == 0 &&
            c->rope_theta > 0.f && c->rms_eps >= 0.f && c->max_block >= 1 && c->max_block <= 16 &&
            c->max_batch >= 1 && c->max_batch <= 256 && c->kv_capacity >= c->max_block &&
            static_cast<long long>(c->max_batch) * c->kv_capacity < (1LL << 31) &&
            ceil_div(c->vocab, 128) <= 65536;
  return ok ? DFLASH_OK : DFLASH_E_CONFIG;
}

size_t dflash_workspace_size(const dflash_config* c) {
  if (dflash_config_check(c) != DFLASH_OK) return 0;
  return layout_of(*c).total;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, dflash_handle** out) {
  if (!cfg || !w || !out) return DFLASH_E_INVAL;
  DFL_TRY(dflash_config_check(cfg));
  const void* globals[] = {w->w_fc, w->g_ctx, w->embed, w->mask_emb, w->g_final, w->lm_head};
  for (const void* p : globals)
    if (!p || !aligned16(p)) return DFLASH_E_INVAL;
  if (!w->layers) return DFLASH_E_INVAL;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    const void* ps[] = {lw.wq, lw.wk, lw.wv, lw.wo, lw.w_gate, lw.w_up, lw.w_down, lw.g_attn, lw.g_mlp};
    for (const void* p : ps)
      if (!p || !aligned16(p)) return DFLASH_E_INVAL;
  }
  if (!get_encoder()) return DFLASH_E_CUDA;
  auto* h = new dflash_handle();
  h->cfg = *cfg;
  h->w = *w;
  h->layers.assign(w->layers, w->layers + cfg->n_layers);
  h->w.layers = h->layers.data();
  h->inject_pass_rows = 16 * nb_for_rows(std::min(cfg->max_batch * cfg->max_block, kMaxPassRows));
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->n_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
      gemv_set_attributes() != 0 || attn_set_attributes() != 0 || attn_tc_set_attributes() != 0) {
    delete h;
    return DFLASH_E_CUDA;
  }
  h->attn_wide = attn_resident_clusters(12);
  const auto& c = *cfg;
  const uint64_t H = c.hidden, d = c.head_dim, I = c.intermediate;
  bool ok = enc2d(&h->m_fc, w->w_fc, static_cast<uint64_t>(c.n_taps) * c.target_hidden, H, 64) &&
            enc2d(&h->m_lm, w->lm_head, H, c.vocab, 64);
  const int L = c.n_layers;
  for (auto* v : {&h->m_wq, &h->m_wk, &h->m_wv, &h->m_wo, &h->m_wg, &h->m_wu, &h->m_wd}) v->resize(L);
  for (int l = 0; l < L && ok; ++l) {
    const dflash_layer_weights& lw = h->layers[l];
    ok = enc2d(&h->m_wq[l], lw.wq, H, c.n_heads * d, 64) && enc2d(&h->m_wk[l], lw.wk, H, c.n_kv_heads * d, 64) &&
         enc2d(&h->m_wv[l], lw.wv, H, c.n_kv_heads * d, 64) && enc2d(&h->m_wo[l], lw.wo, c.n_heads * d, H, 64) &&
         enc2d(&h->m_wg[l], lw.w_gate, H, I, 64) && enc2d(&h->m_wu[l], lw.w_up, H, I, 64) &&
         enc2d(&h->m_wd[l], lw.w_down, I, H, 64);
  }
  if (!ok) {
    delete h;
    return DFLASH_E_CUDA;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle* h) {
  if (!h) return DFLASH_E_INVAL;
  delete h;
  return DFLASH_OK;
}

}  // extern "C"

namespace {

// Shared by both binding calls: records the caches (sequence-major when page_table is null,
// else a pool of layer_rows positions per layer in pages of kPageRows), fills the RoPE
// tables, clears the workspace and encodes the tensor maps over caches and workspace.
int bind_common(dflash_handle* h, void* k_cache, void* v_cache, int layer_rows, const int32_t* page_table,
                int pages_per_seq, int32_t* len, int32_t* last_token, void* workspace, size_t workspace_bytes) {
  const auto& c = h->cfg;
  const WsLayout L = layout_of(c);
  if (workspace_bytes < L.total) return DFLASH_E_CAPACITY;
  h->kc = static_cast<__half*>(k_cache);
  h->vc = static_cast<__half*>(v_cache);
  h->layer_rows = layer_rows;
  h->page_table = page_table;
  h->pages_per_seq = pages_per_seq;
  h->len = len;
  h->last_token = last_token;
  h->ws = static_cast<uint8_t*>(workspace);
  h->L = L;
  if (cudaMemset(workspace, 0, L.total) != cudaSuccess) return DFLASH_E_CUDA;
  // RoPE tables: angle = pos * theta^(-2j/d), computed in double, stored as fp32.
  const int half = c.head_dim / 2;
  std::vector<float> cs(static_cast<size_t>(c.kv_capacity) * half), sn(cs.size());
  for (int p = 0; p < c.kv_capacity; ++p)
    for (int j = 0; j < half; ++j) {
      const double inv = std::pow(static_cast<double>(c.rope_theta), -2.0 * j / c.head_dim);
      const double a = static_cast<double>(p) * inv;
      cs[static_cast<size_t>(p) * half + j] = static_cast<float>(std::cos(a));
      sn[static_cast<size_t>(p) * half + j] = static_cast<float>(std::sin(a));
    }
  if (cudaMemcpy(h->ws + L.rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(h->ws + L.rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return DFLASH_E_CUDA;
  const uint64_t H = c.hidden, d = c.head_dim;
  bool ok = true;
  for (int k = 0; k < 5 && ok; ++k) {
    const uint32_t box = 16u << k;
    ok = enc2d(&h->m_xg[k], h->ws + L.xg, H, 2 * L.R, box) &&
         enc2d(&h->m_cfeat[k], h->ws + L.cfeat, H, 2 * kMaxPassRows, box) &&
         enc2d(&h->m_act[k], h->ws + L.act, c.intermediate, 2 * L.R, box) &&
         enc2d(&h->m_o[k], h->ws + L.o, c.n_heads * d, 2 * L.R, box) &&
         enc2d(&h->m_txg[k], h->ws + L.tgt_xg, c.target_hidden, 2 * L.R, box);
  }
  h->m_kcache.resize(c.n_layers);
  h->m_vcache.resize(c.n_layers);
  h->m_kcache32.resize(c.n_layers);
  h->m_vcache32.resize(c.n_layers);
  const size_t layer_elems = static_cast<size_t>(layer_rows) * c.n_kv_heads * d;
  for (int l = 0; l < c.n_layers && ok; ++l) {
    ok = enc3d_cache(&h->m_kcache[l], h->kc + l * layer_elems, d, c.n_kv_heads, layer_rows) &&
         enc3d_cache(&h->m_vcache[l], h->vc + l * layer_elems, d, c.n_kv_heads, layer_rows) &&
         enc3d_cache(&h->m_kcache32[l], h->kc + l * layer_elems, d, c.n_kv_heads, layer_rows, 32) &&
         enc3d_cache(&h->m_vcache32[l], h->vc + l * layer_elems, d, c.n_kv_heads, layer_rows, 32);
  }
  if (!ok) return DFLASH_E_CUDA;
  h->bound = true;
  return DFLASH_OK;
}

}  // namespace

extern "C" {

int dflash_bind_state(dflash_handle* h, void* k_cache, void* v_cache, int32_t* len, int32_t* last_token,
                      void* workspace, size_t workspace_bytes) {
  if (!h || !k_cache || !v_cache || !len || !last_token || !workspace) return DFLASH_E_INVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) || !aligned16(k_cache) || !aligned16(v_cache))
    return DFLASH_E_INVAL;
  const auto& c = h->cfg;
  return bind_common(h, k_cache, v_cache, c.max_batch * c.kv_capacity, nullptr, 0, len, last_token, workspace,
                     workspace_bytes);
}

int dflash_bind_state_paged(dflash_handle* h, void* k_pool, void* v_pool, int32_t n_pages,
                            const int32_t* page_table, int32_t pages_per_seq, int32_t* len, int32_t* last_token,
                            void* workspace, size_t workspace_bytes) {
  if (!h || !k_pool || !v_pool || !page_table || !len || !last_token || !workspace) return DFLASH_E_INVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned4(page_table))
    return DFLASH_E_INVAL;
  const auto& c = h->cfg;
  if (n_pages < 1 || pages_per_seq < 1 || static_cast<long long>(pages_per_seq) * kPageRows < c.kv_capacity ||
      static_cast<long long>(n_pages) * kPageRows >= (1LL << 31))
    return DFLASH_E_INVAL;
  return bind_common(h, k_pool, v_pool, n_pages * kPageRows, page_table, pages_per_seq, len, last_token, workspace,
                     workspace_bytes);
}

int dflash_inject_ctx(dflash_handle* h, const void* hidden, int32_t rows_per_seq, const int32_t* n_new,
                      int32_t batch, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  if (!hidden || !n_new || !aligned16(hidden) || rows_per_seq < 1 || batch < 1) return DFLASH_E_INVAL;
  if (batch > c.max_batch) return DFLASH_E_CAPACITY;
  const long long total_rows = static_cast<long long>(batch) * rows_per_seq;
  if (total_rows >= (1LL << 31)) return DFLASH_E_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  const int pass_rows = h->inject_pass_rows;
  const int nb = pass_rows / 16;  // a power of two by construction
  const int n_pass = ceil_div(total_rows, pass_rows);
  CUtensorMap m_hidden;
  if (!enc3d_hidden(&m_hidden, hidden, c.target_hidden, total_rows, c.n_taps, pass_rows)) return DFLASH_E_CUDA;
  const int H = c.hidden, d = c.head_dim;
  const int tkv = c.n_kv_heads * d / 128;
  for (int p = 0; p < n_pass; ++p) {
    const int row0 = p * pass_rows;
    GemvParams ph[kMaxPhases]{};
    int np = 0;
    {  // context fusion: F = concat(hidden taps) · Wfcᵀ
      GemvParams& P = ph[np++];
      gemv_common(h, P);
      P.amap[0] = h->m_fc;
      P.n_amaps = 1;
      P.tile_start[0] = 0;
      P.tile_start[1] = H / 128;
      P.T = H / 128;
      P.KB = c.n_taps * c.target_hidden / 64;
      P.bmap = m_hidden;
      P.b3d = 1;
      P.b_kb_per_tap = c.target_hidden / 64;
      P.b_row0 = row0;
      P.grow0 = row0;
      P.out_row0 = 0;
      P.op = OP_FC;
      P.gain = static_cast<const __nv_bfloat16*>(h->w.g_ctx);
      P.yb = h->at<__nv_bfloat16>(h->L.cfeat);
      P.yb_ld = H;
      P.yb_lo = kMaxPassRows;
      P.ss_out = h->at<float>(h->L.ss_fc);
      P.ss_stride = kMaxPassRows;
    }
    for (int l0 = 0; l0 < c.n_layers; l0 += kMaxLayersPerKvLaunch) {  // K/V of every layer
      const int nl = std::min(kMaxLayersPerKvLaunch, c.n_layers - l0);
      GemvParams& P = ph[np++];
      gemv_common(h, P);
      P.n_amaps = 2 * nl;
      for (int i = 0; i < nl; ++i) {
        P.amap[2 * i] = h->m_wk[l0 + i];
        P.amap[2 * i + 1] = h->m_wv[l0 + i];
      }
      for (int i = 0; i <= 2 * nl; ++i) P.tile_start[i] = i * tkv;
      P.T = 2 * nl * tkv;
      P.KB = H / 64;
      P.bmap = h->m_cfeat[nb_index(nb)];
      P.b_row0 = 0;
      P.b_lo = kMaxPassRows;
      P.grow0 = row0;
      P.op = OP_KV;
      P.ss_in = h->at<float>(h->L.ss_fc);
      P.ss_parts = H / 128;
      P.ss_stride = kMaxPassRows;
      P.ss_row0 = 0;
      P.rope_cos = h->at<float>(h->L.rope_cos);
      P.rope_sin = h->at<float>(h->L.rope_sin);
      P.d = d;
      P.kc = h->kc + static_cast<size_t>(l0) * h->layer_rows * c.n_kv_heads * d;
      P.vc = h->vc + static_cast<size_t>(l0) * h->layer_rows * c.n_kv_heads * d;
      P.layer_rows = h->layer_rows;
      P.page_table = h->page_table;
      P.pages_per_seq = h->pages_per_seq;
      P.nkv = c.n_kv_heads;
      P.cap = c.kv_capacity;
      P.max_batch = c.max_batch;
      P.len = h->len;
      P.n_new = n_new;
      P.rows_per_seq = rows_per_seq;
      P.batch = batch;
      P.commit_len = (p == n_pass - 1) && (l0 + nl == c.n_layers);
    }
    DFL_TRY(run_chain(h, ph, np, nb, st));
  }
  return DFLASH_OK;
}

int dflash_draft_block(dflash_handle* h, int32_t batch, int32_t block, int32_t* drafted, float* logits,
                       float* x_trace, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  if (batch < 1 || block < 1 || (block > 1 && !drafted)) return DFLASH_E_INVAL;
  if (!aligned16(logits) || !aligned16(x_trace)) return DFLASH_E_INVAL;  // written 16 bytes at a time
  if (batch > c.max_batch || block > c.max_block) return DFLASH_E_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  const int rows = batch * block;
  const int H = c.hidden, d = c.head_dim, L = c.n_layers, R = h->L.R;
  const int tq = c.n_heads * d / 128, tk = c.n_kv_heads * d / 128;
  const size_t layer_elems = static_cast<size_t>(c.max_batch) * c.kv_capacity * c.n_kv_heads * d;
  {
    EmbedParams E{};
    E.embed = static_cast<const __nv_bfloat16*>(h->w.embed);
    E.mask_emb = static_cast<const __nv_bfloat16*>(h->w.mask_emb);
    E.gain = static_cast<const __nv_bfloat16*>(h->layers[0].g_attn);
    E.last_token = h->last_token;
    E.len = h->len;
    E.x = h->at<float>(h->L.x);
    E.xg = h->at<__nv_bfloat16>(h->L.xg);
    E.xg_lo = R;
    E.ss = h->at<float>(h->L.ss_emb);
    E.trace = x_trace;
    E.err = h->at<int>(h->L.err);
    E.B = block;
    E.H = H;
    E.V = c.vocab;
    E.cap = c.kv_capacity;
    E.tl = tl_take(h, batch * block);
    E.tl_id = h->tl_launch++;
    if (launch_embed(E, batch, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
    note_launch(h, st);
  }
  // Projection phases for a pass of rows [row0, row0 + pass rows).
  auto base = [&](GemvParams& P, int row0, const CUtensorMap& bmap) {
    gemv_common(h, P);
    P.bmap = bmap;
    P.b_row0 = row0;
    P.b_lo = R;  // every draft operand has its low plane R rows down
    P.yb_lo = R;
    P.grow0 = row0;
    P.out_row0 = row0;
    P.ss_row0 = row0;
    P.n_valid = rows;
    P.rows_per_seq = block;
    P.batch = batch;
  };
  auto qkv = [&](GemvParams& P, int l, int row0, int nb) {  // q, k, v with RoPE; block k/v into the cache
    base(P, row0, h->m_xg[nb_index(nb)]);
    P.amap[0] = h->m_wq[l];
    P.amap[1] = h->m_wk[l];
    P.amap[2] = h->m_wv[l];
    P.n_amaps = 3;
    P.tile_start[0] = 0;
    P.tile_start[1] = tq;
    P.tile_start[2] = tq + tk;
    P.tile_start[3] = tq + 2 * tk;
    P.T = tq + 2 * tk;
    P.KB = H / 64;
    P.op = OP_QKV;
    if (l == 0) {
      P.ss_in = h->at<float>(h->L.ss_emb);
      P.ss_parts = 1;
    } else {
      P.ss_in = h->at<float>(h->L.ss_x);
      P.ss_parts = H / 128;
    }
    P.ss_stride = R;
    P.qh = h->at<__half>(h->L.q);
    P.yb_ld = c.n_heads * d;
    P.rope_cos = h->at<float>(h->L.rope_cos);
    P.rope_sin = h->at<float>(h->L.rope_sin);
    P.d = d;
    P.kc = h->kc;
    P.vc = h->vc;
    P.layer_rows = h->layer_rows;
    P.page_table = h->page_table;
    P.pages_per_seq = h->pages_per_seq;
    P.nkv = c.n_kv_heads;
    P.cap = c.kv_capacity;
    P.max_batch = c.max_batch;
    P.layer = l;
    P.len = h->len;
  };
  auto oproj = [&](GemvParams& P, int l, int row0, int nb) {  // x += o · Woᵀ
    base(P, row0, h->m_o[nb_index(nb)]);
    P.amap[0] = h->m_wo[l];
    P.n_amaps = 1;
    P.tile_start[1] = H / 128;
    P.T = H / 128;
    P.KB = c.n_heads * d / 64;
    P.op = OP_RESID;
    P.y = h->at<float>(h->L.x);
    P.y_ld = H;
    P.yb = h->at<__nv_bfloat16>(h->L.xg);
    P.yb_ld = H;
    P.gain = static_cast<const __nv_bfloat16*>(h->layers[l].g_mlp);
    P.ss_out = h->at<float>(h->L.ss_x);
    P.ss_stride = R;
  };
  auto gateup = [&](GemvParams& P, int l, int row0, int nb) {  // act = silu(gate) * up
    base(P, row0, h->m_xg[nb_index(nb)]);
    P.amap[0] = h->m_wg[l];
    P.amap[1] = h->m_wu[l];
    P.n_amaps = 2;
    P.pair_mode = 1;
    P.T = c.intermediate / 64;
    P.KB = H / 64;
    P.op = OP_SWIGLU;
    P.ss_in = h->at<float>(h->L.ss_x);
    P.ss_parts = H / 128;
    P.ss_stride = R;
    P.yb = h->at<__nv_bfloat16>(h->L.act);
    P.yb_ld = c.intermediate;
  };
  auto down = [&](GemvParams& P, int l, int row0, int nb) {  // x += act · W_downᵀ
    base(P, row0, h->m_act[nb_index(nb)]);
    P.amap[0] = h->m_wd[l];
    P.n_amaps = 1;
    P.tile_start[1] = H / 128;
    P.T = H / 128;
    P.KB = c.intermediate / 64;
    P.op = OP_RESID;
    P.y = h->at<float>(h->L.x);
    P.y_ld = H;
    P.yb = h->at<__nv_bfloat16>(h->L.xg);
    P.yb_ld = H;
    P.gain = static_cast<const __nv_bfloat16*>(l + 1 < L ? h->layers[l + 1].g_attn : h->w.g_final);
    P.ss_out = h->at<float>(h->L.ss_x);
    P.ss_stride = R;
    P.trace = x_trace ? x_trace + static_cast<size_t>(l + 1) * rows * H : nullptr;
  };
  auto lmhead = [&](GemvParams& P, int row0, int nb) {  // final norm, LM head, argmax
    base(P, row0, h->m_xg[nb_index(nb)]);
    P.amap[0] = h->m_lm;
    P.n_amaps = 1;
    P.T = ceil_div(c.vocab, 128);
    P.tile_start[1] = P.T;
    P.KB = H / 64;
    P.op = OP_LMHEAD;
    P.ss_in = h->at<float>(h->L.ss_x);
    P.ss_parts = H / 128;
    P.ss_stride = R;
    P.logits = logits;
    P.vocab = c.vocab;
    P.n_out = c.vocab;
    P.best_v = h->at<float>(h->L.best_v);
    P.best_i = h->at<int>(h->L.best_i);
    P.drafted = drafted;
  };
  // Rows are processed in passes of at most kMaxPassRows (one MMA N per pass); each pass
  // runs its chain of projections independently (rows do not interact outside attention).
  auto chain_passes = [&](auto&& build) -> int {
    for (int row0 = 0; row0 < rows; row0 += kMaxPassRows) {
      const int nb = nb_for_rows(std::min(kMaxPassRows, rows - row0));
      GemvParams ph[kMaxPhases]{};
      const int np = build(ph, row0, nb);
      if (np > 0) DFL_TRY(run_chain(h, ph, np, nb, st));
    }
    return DFLASH_OK;
  };
  auto attention = [&](int l) -> int {  // bidirectional attention over injected context + block
    AttnParams A{};
    A.kmap = h->m_kcache[l];
    A.vmap = h->m_vcache[l];
    A.kmap32 = h->m_kcache32[l];
    A.vmap32 = h->m_vcache32[l];
    A.q = h->at<__half>(h->L.q);
    A.o = h->at<__nv_bfloat16>(h->L.o);
    A.o_lo = R;
    A.len = h->len;
    A.page_table = h->page_table;
    A.pages_per_seq = h->pages_per_seq;
    A.n_pages = h->layer_rows / kPageRows;
    A.err = h->at<int>(h->L.err);
    A.B = block;
    A.nq = c.n_heads;
    A.nkv = c.n_kv_heads;
    A.d = d;
    A.cap = c.kv_capacity;
    A.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    // one cluster per (sequence, KV head), splitting its keys over as many SMs as allow one
    // wave: 12 CTAs where that many clusters of 12 fit at once (measured best on GB300 at
    // ctx 2048: 16.5 us against 19.3 us with 8; clusters of 16 ran in two waves), else <= 8
    const int pairs = batch * c.n_kv_heads;
    int split = h->n_sms / pairs;
    split = (split >= 12 && h->attn_wide >= pairs) ? 12 : std::max(1, std::min(8, split));
    A.wait_ns = h->wait_ns;
    A.key_groups = (c.n_heads / c.n_kv_heads <= 4) ? h->attn_key_groups : 1;
    // Clusters of 12 where every pair gets one at once (few sequences: the merge runs in
    // distributed shared memory); otherwise one flat list of every pair's key tiles split
    // evenly over the SMs, which balances ragged and long contexts.
    const bool flat = batch <= kAttnFlatMaxBatch &&
                      (h->attn_mode >= 2 || (h->attn_mode == 0 && h->attn_split == 0 && split < 12));
    if (flat) {
      const int G = std::min(h->n_sms, kMaxCtas);
      A.batch = batch;
      A.part = h->at<float>(h->L.attn_part);
      A.cnt = h->at<int>(h->L.attn_cnt);
      A.tl = tl_take(h, G);
      A.tl_id = h->tl_launch++;
      // the tensor-core kernel where every head pair gets two SMs or more (long contexts:
      // few segment switches, whose pipeline drain it pays); the mma.sync one for many sequences
      const bool tc = attn_tc_supported(A) &&
                      (h->attn_mode == 2 || (h->attn_mode == 0 && batch * c.n_kv_heads <= h->n_sms));
      if ((tc ? launch_attention_flat_tc(A, G, st, h->trace_ev.empty())
              : launch_attention_flat(A, G, st, h->trace_ev.empty())) != 0)
        return DFLASH_E_CUDA;
      note_launch(h, st);
      return DFLASH_OK;
    }
    if (h->attn_split > 0) split = h->attn_split;
    A.tl = tl_take(h, static_cast<long long>(split) * c.n_kv_heads * batch);
    A.tl_id = h->tl_launch++;
    if (launch_attention(A, batch, split, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
    note_launch(h, st);
    return DFLASH_OK;
  };
  // chain sequence: [qkv 0] attn 0 [o 0, gate/up 0, down 0, qkv 1] attn 1 ... [o L-1, ..., LM head]
  DFL_TRY(chain_passes([&](GemvParams* ph, int row0, int nb) {
    qkv(ph[0], 0, row0, nb);
    return 1;
  }));
  for (int l = 0; l < L; ++l) {
    DFL_TRY(attention(l));
    DFL_TRY(chain_passes([&](GemvParams* ph, int row0, int nb) {
      int np = 0;
      oproj(ph[np++], l, row0, nb);
      gateup(ph[np++], l, row0, nb);
      down(ph[np++], l, row0, nb);
      if (l + 1 < L) qkv(ph[np++], l + 1, row0, nb);
      else if (block > 1) lmhead(ph[np++], row0, nb);
      return np;
    }));
  }
  (void)layer_elems;
  return DFLASH_OK;
}

int dflash_verify_greedy(dflash_handle* h, const float* target_logits, const int32_t* drafted, int32_t batch,
                         int32_t block, int32_t* accept_len, int32_t* committed, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  if (!target_logits || !accept_len || !committed || batch < 1 || block < 1 || (block > 1 && !drafted))
    return DFLASH_E_INVAL;
  // the logits are read 16 bytes at a time, the token arrays as 4-byte words
  if (!aligned16(target_logits) || !aligned4(drafted) || !aligned4(accept_len) || !aligned4(committed))
    return DFLASH_E_INVAL;
  if (batch > c.max_batch || block > c.max_block) return DFLASH_E_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  VerifyParams P{};
  P.logits = target_logits;
  P.drafted = drafted;
  P.accept_len = accept_len;
  P.committed = committed;
  P.last_token = h->last_token;
  P.part_v = h->at<float>(h->L.vpart_v);
  P.part_i = h->at<int>(h->L.vpart_i);
  P.seq_cnt = h->at<int>(h->L.seq_cnt);
  P.err = h->at<int>(h->L.err);
  P.B = block;
  P.V = c.vocab;
  int chunks = std::max(1, std::min(kMaxChunks, ceil_div(2LL * h->n_sms, static_cast<long long>(batch) * block)));
  P.chunk_len = static_cast<int>(align_up(static_cast<size_t>(ceil_div(c.vocab, chunks)), 1024));
  P.chunks = ceil_div(c.vocab, P.chunk_len);
  P.tl = tl_take(h, static_cast<long long>(P.chunks) * block * batch);
  P.tl_id = h->tl_launch++;
  if (launch_verify(P, batch, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
  note_launch(h, st);
  return DFLASH_OK;
}

int dflash_verify_sampling(dflash_handle* h, const float* target_logits, const int32_t* drafted,
                           const float* uniforms, float temperature, int32_t batch, int32_t block,
                           int32_t* accept_len, int32_t* committed, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  if (!target_logits || !uniforms || !accept_len || !committed || batch < 1 || block < 1 || (block > 1 && !drafted))
    return DFLASH_E_INVAL;
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return DFLASH_E_INVAL;
  if (!aligned4(target_logits) || !aligned4(uniforms) || !aligned4(drafted) || !aligned4(accept_len) ||
      !aligned4(committed))
    return DFLASH_E_INVAL;
  if (batch > c.max_batch || block > c.max_block) return DFLASH_E_CAPACITY;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  VerifySampleParams P{};
  P.logits = target_logits;
  P.drafted = drafted;
  P.uniforms = uniforms;
  P.inv_temp = 1.f / temperature;
  P.accept_len = accept_len;
  P.committed = committed;
  P.last_token = h->last_token;
  P.part_m = h->at<float>(h->L.vpart_v);
  P.part_s = h->at<float>(h->L.vpart_i);
  P.seq_cnt = h->at<int>(h->L.seq_cnt);
  P.err = h->at<int>(h->L.err);
  P.B = block;
  P.V = c.vocab;
  const int chunks = std::max(1, std::min(kMaxChunks, ceil_div(2LL * h->n_sms, static_cast<long long>(batch) * block)));
  P.chunk_len = static_cast<int>(align_up(static_cast<size_t>(ceil_div(c.vocab, chunks)), 1024));
  P.chunks = ceil_div(c.vocab, P.chunk_len);
  if (launch_verify_sampling(P, batch, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
  note_launch(h, st);
  return DFLASH_OK;
}

int dflash_verify_greedy_hidden(dflash_handle* h, const void* target_hidden, const void* target_gain,
                                const void* target_lm_head, const int32_t* drafted, int32_t batch, int32_t block,
                                int32_t* accept_len, int32_t* committed, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  if (!target_hidden || !target_gain || !target_lm_head || !accept_len || !committed || batch < 1 || block < 1 ||
      (block > 1 && !drafted))
    return DFLASH_E_INVAL;
  if (!aligned16(target_hidden) || !aligned16(target_gain) || !aligned16(target_lm_head) || !aligned4(drafted) ||
      !aligned4(accept_len) || !aligned4(committed))
    return DFLASH_E_INVAL;
  if (batch > c.max_batch || block > c.max_block) return DFLASH_E_CAPACITY;
  if (c.target_hidden > 8192) return DFLASH_E_CONFIG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  const int rows = batch * block, Ht = c.target_hidden, R = h->L.R;
  CUtensorMap m_lm;
  if (!enc2d(&m_lm, target_lm_head, Ht, c.vocab, 64)) return DFLASH_E_CUDA;
  TargetPrepParams T{};
  T.hidden = static_cast<const __nv_bfloat16*>(target_hidden);
  T.gain = static_cast<const __nv_bfloat16*>(target_gain);
  T.xg = h->at<__nv_bfloat16>(h->L.tgt_xg);
  T.xg_lo = R;
  T.ss = h->at<float>(h->L.tgt_ss);
  T.Ht = Ht;
  if (launch_target_prep(T, rows, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
  note_launch(h, st);
  for (int row0 = 0; row0 < rows; row0 += kMaxPassRows) {  // the target's argmax of every row
    const int nb = nb_for_rows(std::min(kMaxPassRows, rows - row0));
    GemvParams P{};
    gemv_common(h, P);
    P.amap[0] = m_lm;
    P.n_amaps = 1;
    P.T = ceil_div(c.vocab, 128);
    P.tile_start[1] = P.T;
    P.KB = Ht / 64;
    P.bmap = h->m_txg[nb_index(nb)];
    P.b_row0 = row0;
    P.b_lo = R;
    P.grow0 = row0;
    P.out_row0 = row0;
    P.n_valid = rows;
    P.op = OP_LMHEAD;
    P.ss_in = h->at<float>(h->L.tgt_ss);
    P.ss_parts = 1;
    P.ss_stride = R;
    P.ss_row0 = row0;
    P.H = Ht;
    P.rows_per_seq = block;
    P.batch = batch;
    P.vocab = c.vocab;
    P.n_out = c.vocab;
    P.best_v = h->at<float>(h->L.best_v);
    P.best_i = h->at<int>(h->L.best_i);
    P.drafted = h->at<int>(h->L.tgt_g);
    P.lm_all_rows = 1;
    DFL_TRY(run_gemv(h, P, nb, st));
  }
  AcceptParams A{};
  A.g = h->at<int>(h->L.tgt_g);
  A.drafted = drafted;
  A.accept_len = accept_len;
  A.committed = committed;
  A.last_token = h->last_token;
  A.batch = batch;
  A.B = block;
  if (launch_accept(A, st, h->trace_ev.empty()) != 0) return DFLASH_E_CUDA;
  note_launch(h, st);
  return DFLASH_OK;
}

int dflash_linear_bf16(dflash_handle* h, const void* W, int32_t n_out, int32_t K, const void* X, int32_t rows,
                       float* Y, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  if (!W || !X || !Y || !aligned16(W) || !aligned16(X) || n_out < 1 || K < 64 || K % 64 || rows < 1)
    return DFLASH_E_INVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  CUtensorMap mw;
  if (!enc2d(&mw, W, K, n_out, 64)) return DFLASH_E_CUDA;
  for (int row0 = 0; row0 < rows; row0 += kMaxPassRows) {
    const int pr = std::min(kMaxPassRows, rows - row0);
    const int nb = nb_for_rows(pr);
    CUtensorMap mx;
    if (!enc2d(&mx, X, K, rows, 16 * nb)) return DFLASH_E_CUDA;
    GemvParams P{};
    gemv_common(h, P);
    P.amap[0] = mw;
    P.n_amaps = 1;
    P.T = ceil_div(n_out, 128);
    P.tile_start[1] = P.T;
    P.KB = K / 64;
    P.bmap = mx;
    P.b_row0 = row0;
    P.grow0 = row0;
    P.out_row0 = row0;
    P.n_valid = rows;
    P.n_out = n_out;
    P.op = OP_PLAIN;
    P.y = Y;
    P.y_ld = n_out;
    DFL_TRY(run_gemv(h, P, nb, st));
  }
  return DFLASH_OK;
}

int dflash_read_device_error(dflash_handle* h, int32_t* flags, int32_t clear, void* stream) {
  if (!h || !flags) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, h->ws + h->L.err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DFLASH_E_CUDA;
  *flags = v;
  if (clear) {
    // The flag, and every arrival counter a kernel that gave up a wait may have left
    // non-zero (split-tile and phase counters, per-sequence verification counters).
    const WsLayout& L = h->L;
    const size_t spans[][2] = {{L.err, 4},
                               {L.tile_cnt, static_cast<size_t>(L.max_tiles) * 4},
                               {L.cta_cnt, 4},
                               {L.seq_cnt, static_cast<size_t>(h->cfg.max_batch) * 4},
                               {L.chain_bar, static_cast<size_t>(kChainSlots) * (kMaxPhases + 4) * 4},
                               {L.attn_cnt, static_cast<size_t>(h->cfg.max_batch) * h->cfg.n_kv_heads * 4}};
    for (const auto& sp : spans)
      if (cudaMemsetAsync(h->ws + sp[0], 0, sp[1], st) != cudaSuccess) return DFLASH_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DFLASH_E_CUDA;
  }
  return DFLASH_OK;
}

int dflash_set_option(dflash_handle* h, int32_t option, int64_t value) {
  if (!h) return DFLASH_E_INVAL;
  switch (option) {
    case DFLASH_OPT_WAIT_LIMIT_NS:
      if (value < 100000 || value > 60000000000LL) return DFLASH_E_INVAL;
      h->wait_ns = static_cast<unsigned long long>(value);
      return DFLASH_OK;
    case DFLASH_OPT_CHAIN_MAX:
      if (value < 1 || value > kMaxPhases) return DFLASH_E_INVAL;
      h->chain_max = static_cast<int>(value);
      return DFLASH_OK;
    case DFLASH_OPT_GEMV_VARIANT:
      if (value < 0 || value > 5) return DFLASH_E_INVAL;
      h->gemv_pref = static_cast<int>(value);
      return DFLASH_OK;
    case DFLASH_OPT_ATTN_SPLIT:
      if (value < 0 || value > 16) return DFLASH_E_INVAL;
      h->attn_split = static_cast<int>(value);
      return DFLASH_OK;
    case DFLASH_OPT_ATTN_KEY_GROUPS:
      if (value < 1 || value > 2) return DFLASH_E_INVAL;
      h->attn_key_groups = static_cast<int>(value);
      return DFLASH_OK;
    case DFLASH_OPT_INJECT_PASS_ROWS:
      if (value != 16 && value != 32 && value != 64 && value != 128 && value != 256) return DFLASH_E_INVAL;
      h->inject_pass_rows = static_cast<int>(value);
      return DFLASH_OK;
    case DFLASH_OPT_ATTN_MODE:
      if (value < 0 || value > 3) return DFLASH_E_INVAL;
      h->attn_mode = static_cast<int>(value);
      return DFLASH_OK;
  }
  return DFLASH_E_INVAL;
}

int dflash_get_option(const dflash_handle* h, int32_t option, int64_t* value) {
  if (!h || !value) return DFLASH_E_INVAL;
  switch (option) {
    case DFLASH_OPT_WAIT_LIMIT_NS: *value = static_cast<int64_t>(h->wait_ns); return DFLASH_OK;
    case DFLASH_OPT_CHAIN_MAX: *value = h->chain_max; return DFLASH_OK;
    case DFLASH_OPT_GEMV_VARIANT: *value = h->gemv_pref; return DFLASH_OK;
    case DFLASH_OPT_ATTN_SPLIT: *value = h->attn_split; return DFLASH_OK;
    case DFLASH_OPT_ATTN_KEY_GROUPS: *value = h->attn_key_groups; return DFLASH_OK;
    case DFLASH_OPT_INJECT_PASS_ROWS: *value = h->inject_pass_rows; return DFLASH_OK;
    case DFLASH_OPT_ATTN_MODE: *value = h->attn_mode; return DFLASH_OK;
  }
  return DFLASH_E_INVAL;
}

int dflash_selftest_timeout(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_E_INVAL;
  if (!h->bound) return DFLASH_E_STATE;
  const auto& c = h->cfg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  call_begin(h, st);
  // Two plain projections of the residual scratch through the output projection of layer
  // 0 (Y = xg · Woᵀ into the residual scratch, which the next draft rewrites before use).
  // Phase 1 waits for a barrier count one above the grid size, which no CTA reaches.
  GemvParams P{};
  gemv_common(h, P);
  P.amap[0] = h->m_wo[0];
  P.n_amaps = 1;
  P.T = c.hidden / 128;
  P.tile_start[1] = P.T;
  P.KB = c.n_heads * c.head_dim / 64;
  P.bmap = h->m_o[0];
  P.op = OP_PLAIN;
  P.n_valid = 16;
  P.n_out = c.hidden;
  P.y = h->at<float>(h->L.x);
  P.y_ld = c.hidden;
  GemvChain C{};
  const int v = gemv_variant(1, h->gemv_pref);
  const int ks = gemv_variant_ksub(v);
  if (P.KB % ks) return DFLASH_E_CONFIG;
  C.ph[0] = P;
  C.ph[0].KB /= ks;
  C.ph[1] = C.ph[0];
  C.n_phases = 2;
  C.bar = h->at<int>(h->L.chain_bar) + h->chain_slot * (kMaxPhases + 4);
  h->chain_slot = (h->chain_slot + 1) % kChainSlots;
  C.exit_cnt = C.bar + kMaxPhases;
  C.wait_ns = h->wait_ns;
  C.bar_extra = 1;
  const int e = launch_gemv(C, v, std::min(h->n_sms, kMaxCtas), st, false);
  note_launch(h, st);
  return e == 0 ? DFLASH_OK : DFLASH_E_CUDA;
}

int32_t dflash_last_launch_count(const dflash_handle* h) { return h ? h->last_launches : 0; }

int dflash_timeline(dflash_handle* h, void* records, int64_t n_records) {
  if (!h || n_records < 0 || (n_records > 0 && !records)) return DFLASH_E_INVAL;
  h->tl_buf = n_records > 0 ? static_cast<unsigned long long*>(records) : nullptr;
  h->tl_cap = n_records;
  h->tl_next = 0;
  h->tl_launch = 0;
  return DFLASH_OK;
}

int64_t dflash_timeline_used(const dflash_handle* h) { return h ? h->tl_next : 0; }

int dflash_trace_events(dflash_handle* h, void* const* events, int32_t n_events) {
  if (!h || n_events < 0 || (n_events > 0 && !events)) return DFLASH_E_INVAL;
  h->trace_ev.clear();
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return DFLASH_E_INVAL;
    h->trace_ev.push_back(static_cast<cudaEvent_t>(events[i]));
  }
  return DFLASH_OK;
}

const char* dflash_status_string(int s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_E_INVAL: return "invalid argument";
    case DFLASH_E_CONFIG: return "unsupported drafter shape";
    case DFLASH_E_CAPACITY: return "capacity exceeded";
    case DFLASH_E_CUDA: return "CUDA error";
    case DFLASH_E_STATE: return "state not bound";
  }
  return "unknown status";
}

int dflash_synth_plant(float* logits, const int32_t* drafted, const uint8_t* plant_masks, int32_t n_steps,
                       const int32_t* step_counter, int32_t batch, int32_t block, int32_t vocab, float bump,
                       int32_t* saved, void* stream) {
  if (!logits || !plant_masks || !step_counter || !saved || n_steps < 1 || batch < 1 || block < 1 || vocab < 1 ||
      (block > 1 && !drafted))
    return DFLASH_E_INVAL;
  if (static_cast<long long>(batch) * block * vocab >= (1LL << 31)) return DFLASH_E_CAPACITY;
  return launch_plant(logits, drafted, plant_masks, n_steps, step_counter, batch, block, vocab, bump, saved,
                      static_cast<cudaStream_t>(stream)) == 0
             ? DFLASH_OK
             : DFLASH_E_CUDA;
}

int dflash_synth_unplant(float* logits, int32_t* step_counter, int32_t n_steps, int32_t batch, int32_t block,
                         const int32_t* saved, void* stream) {
  if (!logits || !step_counter || !saved || n_steps < 1 || batch < 1 || block < 1) return DFLASH_E_INVAL;
  return launch_unplant(logits, step_counter, n_steps, batch, block, saved, static_cast<cudaStream_t>(stream)) == 0
             ? DFLASH_OK
             : DFLASH_E_CUDA;
}

}  // extern "C"
