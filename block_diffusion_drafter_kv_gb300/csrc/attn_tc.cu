// Flat key-split block attention on the tcgen05 tensor cores (sm_103a), for head dim 128,
// GQA groups of 4 query heads and an even number of KV heads: the path for many or long
// contexts, where the mma.sync tile loop (every warp reading the whole K/V tile through
// ldmatrix) bounds the flat split.
//
// Two KV heads of a sequence (2h, 2h+1: a "head pair") are processed together, so that the
// 128 rows of an M = 128 MMA are all real: rows 0-63 are head 2h's 4 query heads x 16 block
// slots, rows 64-127 head 2h+1's. The key tiles of every (sequence, head pair), in
// (sequence, pair) order, form one list cut into equal contiguous ranges, one per CTA; a
// pair inside one range is written by its CTA, a pair cut between CTAs is merged by the last
// of them to arrive, in CTA order (as in attn_flat_kernel).
//
// Per step (32 keys of both heads; K and V fp16, staged by TMA in boxes of 32 positions with
// the 128-byte swizzle, the two heads' keys stacked into 64-key operands; a 4-deep ring):
//   S  = Q Kᵀ  : tcgen05.mma kind::f16, M = 128, N = 64 keys, K = 128 dims; fp32 in TMEM
//                (three buffers: the issuer runs two steps ahead). Row r only uses its own
//                head's 32 columns.
//   softmax    : four warps, one query row per thread: the row's 32 scores from TMEM, the
//                running max (log2 units) and sum, P = exp2(S - m) as fp16 into shared
//                memory (two buffers), where the other head's 32 columns of the row stay zero.
//   O += P V   : tcgen05.mma, M = 128, N = 128 dims, K = 64 keys, V read MN-major (its rows
//                are keys with the dims contiguous), accumulated in TMEM over the segment;
//                the zero blocks of P keep each head's rows to its own values.
//   rescale    : a row's probabilities are taken against a reference max that moves only
//                when the tile max exceeds it by more than 8 (log2 units; P then stays
//                <= 256, exact enough in fp16); then that row of O in TMEM and its sum are
//                scaled by exp2(old - new), after the PVs issued so far have completed.
// Roles: warps 0-3 softmax/output, warp 4 lane 0 MMA issuer (up to two QKᵀ ahead of the PVs
// within a segment), warp 5 lane 0 TMA producer. Every wait is bounded, none waits for a phase
// older than the last its barrier can have completed, and the softmax warps take every wait
// and every exit together (warp-collective TMEM accesses never diverge).
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int TKT = 32;             // keys per head per step
constexpr int TST = 4;              // K/V ring stages
constexpr int TD = 128;             // head dim
constexpr int TNW = 4;              // query heads per KV head
constexpr int TR = 2 * TNW * 16;    // rows: two KV heads x 4 query heads x 16 slots = 128
constexpr int TKB = 2 * TKT * 128;  // one 64-dim box of the two heads' keys: 64 rows x 128 B
constexpr int TTILE = 4 * TKB;      // K boxes (dims 0-63, 64-127), then V boxes
constexpr int kTcMaxBatch = 1024;   // sequences per launch (shared-memory prefix table)
// shared memory (offsets from the 1024-aligned base)
constexpr int Q_OFF = 0;                  // 128 rows x 128 dims fp16: two 64-dim boxes of 16 KB
constexpr int P_OFF = 32768;              // two buffers of 128 rows x 64 keys fp16 (16 KB each)
constexpr int RING_OFF = 65536;           // TST x (K box 0, K box 1, V box 0, V box 1)
constexpr int BAR_OFF = RING_OFF + TST * TTILE;
// mbarriers: full[TST], empty[TST], sready[NS], sfree[NS], pready[2], pvready[2], qready, mdone
constexpr int NS = 3;  // S buffers in TMEM
constexpr int NBARS = 2 * TST + 2 * NS + 6;
constexpr int FLAG_OFF = BAR_OFF + NBARS * 8;     // [0] abort, [1] merging, [2] sharers, [3] rank, [4] tmem base
constexpr int CS_OFF = FLAG_OFF + 32;             // merge: contributor slots [kMaxCtas]
constexpr int PRE_OFF = CS_OFF + kMaxCtas * 4;    // tiles per head before each sequence [batch + 1]
constexpr uint32_t S_COL = 0, O_COL = 256;        // TMEM columns: S buffers at 0, 64, 128; O at 256
constexpr float kRescale = 8.f;                   // log2 growth of a row max that moves its reference

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, A K-major, B K-major
// or MN-major, M x N.
constexpr uint32_t idesc_f16_f32(int M, int N, bool b_mn) {
  return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t IDESC_QK = idesc_f16_f32(128, 2 * TKT, false);
constexpr uint32_t IDESC_PV = idesc_f16_f32(128, TD, true);

// Shared-memory descriptor of an MN-major operand written by TMA with the 128-byte swizzle:
// 128-byte rows of 64 consecutive MN elements, one row per K index; 8 K rows form a
// 1024-byte swizzle atom (stride byte offset), and the next 64 MN elements sit `mn_stride`
// bytes further on (leading byte offset). Version 1, layout "128B swizzle".
DEV uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

DEV long long tc_begin(int c, long long T, int G) { return static_cast<long long>(c) * T / G; }
DEV int tc_cta_of(long long u, long long T, int G) { return static_cast<int>(((u + 1) * G + T - 1) / T) - 1; }

// Byte offset of 16-byte chunk `ch` of row `r` in a 128-byte-swizzled box.
DEV uint32_t sw128(int r, int ch) { return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4)); }

// 2^x by the multi-function unit's approximation (relative error about 2^-22, well inside
// the fp16 rounding the probabilities get next).
DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

DEV void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace

__global__ void __launch_bounds__(192, 1) attn_flat_tc_kernel(const __grid_constant__ AttnParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>(blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_ATTN) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  uint64_t* full = bars;
  uint64_t* empty = bars + TST;
  uint64_t* sready = bars + 2 * TST;
  uint64_t* sfree = sready + NS;
  uint64_t* pready = sfree + NS;
  uint64_t* pvready = pready + 2;
  uint64_t* qready = pvready + 2;
  uint64_t* mdone = qready + 1;
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + FLAG_OFF);
  int* s_cs = reinterpret_cast<int*>(smem + CS_OFF);
  int* s_pre = reinterpret_cast<int*>(smem + PRE_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int batch = P.batch, B = P.B, nq = P.nq;
  const int npair = P.nkv / 2;  // head pairs per sequence
  const uint64_t WL = P.wait_ns;

  // ---- set-up: tiles per sequence (len is final here: the kernel before this one, the
  // Q/K/V projection, starts only after this step's injection has completed), barriers, the
  // zero off-diagonal blocks of P
  for (int s = threadIdx.x; s < batch; s += blockDim.x) {
    int nk = __ldcg(P.len + s) + B;
    if (nk > P.cap) nk = P.cap;
    s_pre[s + 1] = (nk + TKT - 1) / TKT;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < TST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    for (int b = 0; b < NS; ++b) {
      mbar_init(&sready[b], 1);
      mbar_init(&sfree[b], TR);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pready[b], TR);
      mbar_init(&pvready[b], 1);
    }
    mbar_init(qready, TR);
    mbar_init(mdone, 1);
    s_flag[0] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 160) {
    tma_prefetch_desc(&P.kmap32);
    tma_prefetch_desc(&P.vmap32);
  }
  {  // in both P buffers rows 0-63 never hold keys 32-63 (chunks 4-7), rows 64-127 never 0-31
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int k = threadIdx.x; k < 2 * 128 * 4; k += blockDim.x) {
      const int buf = k >> 9, r = (k >> 2) & 127, ch = (r < 64 ? 4 : 0) + (k & 3);
      *reinterpret_cast<uint4*>(smem + P_OFF + buf * 16384 + sw128(r, ch)) = z;
    }
    fence_async_shared();
  }
  if (warp == 4) tmem_alloc(reinterpret_cast<uint32_t*>(smem + FLAG_OFF + 16), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + FLAG_OFF + 16);
  if (threadIdx.x == 0) {
    s_pre[0] = 0;
    for (int s = 0; s < batch; ++s) s_pre[s + 1] += s_pre[s];
  }
  __syncthreads();

  const long long T = static_cast<long long>(npair) * s_pre[batch];
  const int G = gridDim.x, c = blockIdx.x;
  const long long T0 = tc_begin(c, T, G);
  const int n = static_cast<int>(tc_begin(c + 1, T, G) - T0);
  // flat step u -> sequence s, head pair g2, tile t of the pair, the pair's tile count nt
  auto locate = [&](long long u, int& s, int& g2, int& t, int& nt) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(npair) * s_pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
    nt = s_pre[s + 1] - s_pre[s];
    const long long r = u - static_cast<long long>(npair) * s_pre[s];
    g2 = static_cast<int>(r / nt);
    t = static_cast<int>(r - static_cast<long long>(g2) * nt);
  };
  // a cursor over the list, advanced one step at a time
  struct Cursor {
    int s, g2, t, nt;
  };
  auto advance = [&](Cursor& q) {  // true when the new step is a pair's first tile
    if (++q.t == q.nt) {
      q.t = 0;
      if (++q.g2 == npair) {
        q.g2 = 0;
        ++q.s;
        if (q.s < batch) q.nt = s_pre[q.s + 1] - s_pre[q.s];
      }
      return true;
    }
    return false;
  };
  const uint64_t kv_pol = T * TTILE > (16ll << 20) ? policy_evict_first() : policy_evict_last();

  if (warp == 5) {
    // ------------------------------------------------------------------ TMA producer
    auto issue = [&](int j, int s, int g2, int t) {
      const int st = j % TST;
      uint8_t* base = smem + RING_OFF + st * TTILE;
      int row = s * P.cap + t * TKT;
      if (P.page_table) {  // a page holds kPageRows positions: two steps
        const int page = __ldcg(P.page_table + static_cast<size_t>(s) * P.pages_per_seq + t / (kPageRows / TKT));
        if (page < 0 || page >= P.n_pages) raise_flag(P.err, kDevCapacity);
        row = (page < 0 || page >= P.n_pages) ? 0 : page * kPageRows + (t % (kPageRows / TKT)) * TKT;
      }
      mbar_arrive_expect_tx(&full[st], TTILE);
      for (int hh = 0; hh < 2; ++hh)
        for (int b = 0; b < TD / 64; ++b) {
          tma_load_3d(base + b * TKB + hh * (TKT * 128), &P.kmap32, &full[st], b * 64, 2 * g2 + hh, row, kv_pol);
          tma_load_3d(base + 2 * TKB + b * TKB + hh * (TKT * 128), &P.vmap32, &full[st], b * 64, 2 * g2 + hh, row,
                      kv_pol);
        }
    };
    const int pre = n < TST ? n : TST;
    if (lane == 0)  // tiles entirely below len do not depend on the previous kernel
      for (int j = 0; j < pre; ++j) {
        int s, g2, t, nt;
        locate(T0 + j, s, g2, t, nt);
        if ((t + 1) * TKT <= __ldcg(P.len + s)) issue(j, s, g2, t);
      }
    __syncwarp();
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0) {
      tl_stamp(tl, 5);
      for (int j = 0; j < pre; ++j) {
        int s, g2, t, nt;
        locate(T0 + j, s, g2, t, nt);
        if ((t + 1) * TKT > __ldcg(P.len + s)) issue(j, s, g2, t);
      }
      int issued = pre;
      Cursor q{0, 0, 0, 1};
      if (pre < n) locate(T0 + pre, q.s, q.g2, q.t, q.nt);
      uint64_t t_blocked = 0;  // timeline: time waiting for a free stage
      for (int j = pre; j < n; ++j) {
        const uint64_t tw = tl ? globaltimer_ns() : 0;
        if (s_flag[0] || !mbar_wait(&empty[j % TST], ((j / TST) - 1) & 1, WL)) {
          if (!s_flag[0]) raise_flag(P.err, kDevTimeout);
          s_flag[0] = 1;
          break;
        }
        if (tl) t_blocked += globaltimer_ns() - tw;
        issue(j, q.s, q.g2, q.t);
        ++issued;
        advance(q);
      }
      if (tl) tl[10] = t_blocked;
      // every copy issued has landed before the CTA may exit (the last TST may not have been
      // consumed after an abandoned wait; earlier ones were, or their stage was not reused)
      for (int k = issued > TST ? issued - TST : 0; k < issued; ++k)
        if (!mbar_wait(&full[k % TST], (k / TST) & 1, WL)) {
          raise_flag(P.err, kDevTimeout);
          break;
        }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA issuer
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0) {
      auto qk = [&](int i) {  // S[i % NS] = Q [K of both heads]ᵀ (its inputs are ready)
        const int st = i % TST, b = i % NS;
        tc_fence_after();
        const uint32_t q0 = smem_u32(smem + Q_OFF), k0 = smem_u32(smem + RING_OFF + st * TTILE);
#pragma unroll
        for (int kk = 0; kk < TD / 16; ++kk) {
          const uint32_t box = kk >> 2, w = (kk & 3) * 32;
          tc_mma_bf16(tmem + S_COL + b * (2 * TKT), smem_desc_k_sw128(q0 + box * 16384 + w),
                      smem_desc_k_sw128(k0 + box * TKB + w), IDESC_QK, kk > 0 ? 1u : 0u);
        }
        tc_commit(&sready[b]);
      };
      auto pv = [&](int i, bool seg_first) {  // O (+)= P [V of both heads]; a segment's first tile starts O
        const int st = i % TST;
        tc_fence_after();
        const uint32_t p0 = smem_u32(smem + P_OFF + (i & 1) * 16384);
        const uint32_t v0 = smem_u32(smem + RING_OFF + st * TTILE + 2 * TKB);
#pragma unroll
        for (int kk = 0; kk < 2 * TKT / 16; ++kk)
          tc_mma_bf16(tmem + O_COL, smem_desc_k_sw128(p0 + kk * 32), smem_desc_mn_sw128(v0 + kk * 2048, TKB), IDESC_PV,
                      (kk > 0 || !seg_first) ? 1u : 0u);
        tc_commit(&pvready[i & 1]);
        tc_commit(&empty[st]);
      };
      // Issue each MMA as soon as its inputs are ready, polling both (a QKᵀ waits for its
      // K/V stage, its S buffer and, at a segment's start, the new Q; a PV for its P), so
      // that neither waits behind the other's dependency. Bounded: no progress for the wait
      // limit abandons the loop.
      Cursor q{0, 0, 0, 1};
      if (n > 0) locate(T0, q.s, q.g2, q.t, q.nt);
      int nqk = 0, npv = 0, seg = -1;
      bool first_of[NS] = {false, false, false};
      uint64_t t_idle = globaltimer_ns();
      uint64_t t_idle_sum = 0, t_prev = globaltimer_ns();  // timeline: time with nothing to issue
      while (npv < n) {
        bool moved = false;
        if (nqk < n && nqk <= npv + (NS - 1)) {
          const bool start = nqk == 0 || q.t == 0;
          if (mbar_try_wait(&full[nqk % TST], (nqk / TST) & 1) &&
              (nqk < NS || mbar_try_wait(&sfree[nqk % NS], ((nqk / NS) - 1) & 1)) &&
              (!start || mbar_try_wait(qready, (seg + 1) & 1))) {
            qk(nqk);
            first_of[nqk % NS] = start;
            if (start) ++seg;
            if (nqk + 1 < n) advance(q);
            ++nqk;
            moved = true;
          }
        }
        if (npv < nqk && mbar_try_wait(&pready[npv & 1], (npv >> 1) & 1)) {
          pv(npv, first_of[npv % NS]);
          ++npv;
          moved = true;
        }
        if (moved) {
          const uint64_t now = globaltimer_ns();
          if (tl && now - t_prev > 200) t_idle_sum += now - t_prev;
          t_prev = t_idle = now;
        } else if (s_flag[0] || globaltimer_ns() - t_idle > WL) {
          if (!s_flag[0]) raise_flag(P.err, kDevTimeout);
          s_flag[0] = 1;
          break;
        }
      }
      if (tl) tl[11] = t_idle_sum;
      tc_commit(mdone);
      if (!mbar_wait(mdone, 0, WL)) raise_flag(P.err, kDevTimeout);
    }
  } else {
    // ------------------------------------------------------------------ softmax / output (rows 0-127)
    pdl_wait();
    pdl_launch_dependents();
    const int r = threadIdx.x;                    // row: head of the pair r / 64, query head
    const int hh = r >> 6, hw = (r >> 4) & 3, slot = r & 15;  // (r / 16) % 4 of its group, slot r % 16
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t orow = tmem + lane_base + O_COL;
    const size_t slot_floats = static_cast<size_t>(TR) * (TD + 4);
    // Waits here are warp-uniform (a warp goes on only if every lane's wait succeeded), so the
    // warp-collective TMEM accesses that follow never diverge; after an abandoned wait the
    // four warps leave together at the next softmax-warp barrier.
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      bool lane_ok = ok && !s_flag[0];
      if (lane_ok && !mbar_wait(bar, parity, WL)) {
        raise_flag(P.err, kDevTimeout);
        s_flag[0] = 1;
        lane_ok = false;
      }
      ok = __all_sync(0xffffffffu, lane_ok);
      return ok;
    };
    auto agree = [&]() {
      named_bar_sync(1, TR);
      ok = ok && !s_flag[0];
      return ok;
    };
    bool merged = false;
    uint64_t t_ws = 0, t_wpv = 0;  // timeline (row 0): time waiting for S, and for a PV
    for (int j = 0; j < n && ok;) {
      int s, g2, ta, nt;
      locate(T0 + j, s, g2, ta, nt);
      const int seg = min(n - j, nt - ta);
      const bool whole = ta == 0 && seg == nt;
      int nkeys = __ldcg(P.len + s) + B;
      if (nkeys > P.cap) nkeys = P.cap;
      const int h = (2 * g2 + hh) * TNW + hw;  // this row's query head
      // this row of Q (fp16, post-RoPE) into both 64-dim boxes; rows of unused slots are zero
      {
        const uint4* src = reinterpret_cast<const uint4*>(P.q + (static_cast<size_t>(s) * B + slot) * nq * TD +
                                                          static_cast<size_t>(h) * TD);
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint4 v = slot < B ? __ldcg(src + ch) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(smem + Q_OFF + (ch >> 3) * 16384 + sw128(r, ch & 7)) = v;
        }
        fence_async_shared();
        mbar_arrive(qready);
      }
      float m = -INFINITY, l = 0.f;  // reference max (log2 units) and the row sum against it
      for (int i = j; i < j + seg && ok; ++i) {
        const int b = i & 1, sb = i % NS;
        const uint64_t tw0 = (tl && r == 0) ? globaltimer_ns() : 0;
        if (!wait(&sready[sb], (i / NS) & 1)) break;
        if (tl && r == 0) t_ws += globaltimer_ns() - tw0;
        if (i == 0 && r == 0) tl_stamp(tl, 6);
        tc_fence_after();
        float sc[TKT];
        {
          uint32_t u[TKT / 16][16];
#pragma unroll
          for (int c16 = 0; c16 < TKT / 16; ++c16)
            tmem_ld16_nw(tmem + lane_base + S_COL + sb * (2 * TKT) + hh * TKT + c16 * 16, u[c16]);
          tmem_wait_ld();
#pragma unroll
          for (int c16 = 0; c16 < TKT / 16; ++c16)
#pragma unroll
            for (int k = 0; k < 16; ++k) sc[c16 * 16 + k] = __uint_as_float(u[c16][k]);
        }
        tc_fence_before();
        mbar_arrive(&sfree[sb]);
        const int key0 = (ta + i - j) * TKT;
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < TKT; ++k) {
          sc[k] = key0 + k < nkeys ? sc[k] * P.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[k]);
        }
        const bool need = i != j && mx > m + kRescale;
        if (i == j) m = mx;  // the segment's first tile: O starts from this tile's PV
        if (__any_sync(0xffffffffu, need)) {
          // a row's reference moves: scale that row of O and its sum by exp2(m - mx), once the
          // PVs issued so far have completed; the warp's other rows scale by 1
          if (!wait(&pvready[(i - 1) & 1], ((i - 1) >> 1) & 1)) break;
          tc_fence_after();
          const float corr = need ? fast_exp2(m - mx) : 1.f;
#pragma unroll
          for (int c16 = 0; c16 < TD / 16; ++c16) {
            uint32_t u[16];
            tmem_ld16_nw(orow + c16 * 16, u);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * corr);
            tmem_st16(orow + c16 * 16, u);
          }
          tmem_wait_st();
          if (need) {
            l *= corr;
            m = mx;
          }
        }
        // P buffer b was last read by the PV of step i - 2
        const uint64_t tw1 = (tl && r == 0) ? globaltimer_ns() : 0;
        if (i >= 2 && !wait(&pvready[b], ((i - 2) >> 1) & 1)) break;
        if (tl && r == 0) t_wpv += globaltimer_ns() - tw1;
        float ls = 0.f;
        uint8_t* prow = smem + P_OFF + b * 16384;
#pragma unroll
        for (int ch = 0; ch < TKT / 8; ++ch) {
          __half2 hv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p0 = fast_exp2(sc[ch * 8 + 2 * k] - m), p1 = fast_exp2(sc[ch * 8 + 2 * k + 1] - m);
            ls += p0 + p1;
            hv[k] = __floats2half2_rn(p0, p1);
          }
          *reinterpret_cast<uint4*>(prow + sw128(r, hh * (TKT / 8) + ch)) = *reinterpret_cast<const uint4*>(hv);
        }
        l += ls;
        fence_async_shared();
        tc_fence_before();
        mbar_arrive(&pready[b]);
      }
      if (!agree()) break;
      // the segment's O, once its last PV has completed
      float o[TD];
      {
        wait(&pvready[(j + seg - 1) & 1], ((j + seg - 1) >> 1) & 1);
        if (!agree()) break;
        tc_fence_after();
#pragma unroll
        for (int c16 = 0; c16 < TD / 16; ++c16) {
          uint32_t u[16];
          tmem_ld16_nw(orow + c16 * 16, u);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) o[c16 * 16 + k] = __uint_as_float(u[k]);
        }
        tc_fence_before();
      }
      // ---- this CTA's part of the pair
      if (whole) {
        if (slot < B) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16* dst = P.o + (static_cast<size_t>(s) * B + slot) * nq * TD + static_cast<size_t>(h) * TD;
#pragma unroll
          for (int c8 = 0; c8 < TD / 8; ++c8) {
            __nv_bfloat162 hp[4], lp[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float v0 = o[c8 * 8 + 2 * k] * inv, v1 = o[c8 * 8 + 2 * k + 1] * inv;
              hp[k] = __floats2bfloat162_rn(v0, v1);
              const float2 f = __bfloat1622float2(hp[k]);
              lp[k] = __floats2bfloat162_rn(v0 - f.x, v1 - f.y);
            }
            *reinterpret_cast<uint4*>(dst + c8 * 8) = *reinterpret_cast<const uint4*>(hp);
            *reinterpret_cast<uint4*>(dst + static_cast<size_t>(P.o_lo) * nq * TD + c8 * 8) =
                *reinterpret_cast<const uint4*>(lp);
          }
        }
      } else {
        const long long base_u = static_cast<long long>(npair) * s_pre[s] + static_cast<long long>(g2) * nt;
        float* slot_p = P.part + (2 * static_cast<size_t>(c) + (j == 0 ? 0 : 1)) * slot_floats;
        if (slot < B) {
#pragma unroll
          for (int d4 = 0; d4 < TD / 4; ++d4)
            __stcg(reinterpret_cast<float4*>(slot_p + static_cast<size_t>(r) * TD + d4 * 4),
                   make_float4(o[4 * d4], o[4 * d4 + 1], o[4 * d4 + 2], o[4 * d4 + 3]));
          __stcg(reinterpret_cast<float4*>(slot_p + static_cast<size_t>(TR) * TD + r * 4), make_float4(m, l, 0.f, 0.f));
        }
        named_bar_sync(1, TR);
        // Count this part in. The CTAs whose last segment this pair is (the first CTA of the
        // pair and those wholly inside it: they finish together, at the ends of their
        // ranges) then wait for every part and share the merge. The pair's last CTA, whose
        // range runs on, writes its part early and does not wait.
        const bool sharer = j + seg == n;
        const int c_first = tc_cta_of(base_u, T, G), c_last = tc_cta_of(base_u + nt - 1, T, G);
        if (r == 0) {
          __threadfence();
          int n_c = 0, n_sh = 0, rank = 0;
          for (int cc = c_first; cc <= c_last; ++cc) {
            const long long b0 = tc_begin(cc, T, G), b1 = tc_begin(cc + 1, T, G);
            if (b1 == b0) continue;
            ++n_c;
            if (b1 <= base_u + nt) {
              if (cc < c) ++rank;
              ++n_sh;
            }
          }
          int* cnt = P.cnt + s * npair + g2;
          asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(cnt) : "memory");
          int go = 1;
          if (sharer) {
            // bounded: every part is written before its CTA waits, and a CTA waits only for
            // CTAs of this pair, whose later waits (if any) are for CTAs after them
            const uint64_t t0w = globaltimer_ns();
            int v;
            for (;;) {
              asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
              if (v >= n_c) break;
              if (globaltimer_ns() - t0w > WL) break;
              __nanosleep(64);
            }
            if (v < n_c) {
              raise_flag(P.err, kDevTimeout);
              s_flag[0] = 1;
              go = 0;
            } else if (atomicAdd(cnt, 1) == n_c + n_sh - 1) {
              *cnt = 0;  // every sharer is past the wait: clear for the next launch
            }
          }
          s_flag[1] = sharer && go;
          s_flag[2] = n_sh;
          s_flag[3] = rank;
        }
        named_bar_sync(1, TR);
        if (s_flag[1]) {
          if (r == 0 && !merged) tl_stamp(tl, 8);
          merged = true;
          // combine the parts in CTA order: out = sum_c exp2(m_c - M) o_c / sum_c exp2(m_c - M) l_c;
          // this CTA takes its share of the 128 rows x 8 blocks of 16 dims
          const int nk = c_last - c_first + 1;
          for (int k = r; k < nk; k += TR) {
            const int cc = c_first + k;
            const long long b0 = tc_begin(cc, T, G);
            s_cs[k] = tc_begin(cc + 1, T, G) > b0 ? 2 * cc + (b0 >= base_u ? 0 : 1) : -1;
          }
          named_bar_sync(1, TR);
          const int n_sh = s_flag[2], rank = s_flag[3];
          constexpr int ITEMS = TR * (TD / 16);
          const int i0 = rank * ITEMS / n_sh, i1 = (rank + 1) * ITEMS / n_sh;
          for (int it = i0 + r; it < i1; it += TR) {
            const int rr = it / (TD / 16), d = (it % (TD / 16)) * 16;
            const int sl2 = rr & 15;
            if (sl2 >= B) continue;
            const int hrow = (2 * g2 + (rr >> 6)) * TNW + ((rr >> 4) & 3);
            // the row's max and normaliser, 8 contributors' loads in flight
            float M = -INFINITY, den = 0.f;
            for (int k0 = 0; k0 < nk; k0 += 8) {
              float2 ml[8];
#pragma unroll
              for (int q2 = 0; q2 < 8; ++q2) {
                const int sl = k0 + q2 < nk ? s_cs[k0 + q2] : -1;
                ml[q2] = sl < 0 ? make_float2(-INFINITY, 0.f)
                                : __ldcg(reinterpret_cast<const float2*>(P.part + sl * slot_floats +
                                                                         static_cast<size_t>(TR) * TD + rr * 4));
              }
#pragma unroll
              for (int q2 = 0; q2 < 8; ++q2) {
                if (ml[q2].x == -INFINITY) continue;
                if (ml[q2].x > M) {
                  den = den * exp2f(M - ml[q2].x) + ml[q2].y;
                  M = ml[q2].x;
                } else {
                  den += ml[q2].y * exp2f(ml[q2].x - M);
                }
              }
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            float acc[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) acc[q] = 0.f;
            for (int k0 = 0; k0 < nk; k0 += 4) {  // 4 contributors' loads in flight, added in order
              float mc[4];
              float4 pv4[4][4];
#pragma unroll
              for (int q2 = 0; q2 < 4; ++q2) {
                const int sl = k0 + q2 < nk ? s_cs[k0 + q2] : -1;
                const float* sp = P.part + (sl < 0 ? 0 : sl) * slot_floats;
                mc[q2] = sl < 0 ? -INFINITY : __ldcg(sp + static_cast<size_t>(TR) * TD + rr * 4);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  pv4[q2][q] = sl < 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                                      : __ldcg(reinterpret_cast<const float4*>(sp + static_cast<size_t>(rr) * TD + d + 4 * q));
              }
#pragma unroll
              for (int q2 = 0; q2 < 4; ++q2) {
                const float wc = mc[q2] == -INFINITY ? 0.f : exp2f(mc[q2] - M) * inv;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  acc[4 * q] += wc * pv4[q2][q].x;
                  acc[4 * q + 1] += wc * pv4[q2][q].y;
                  acc[4 * q + 2] += wc * pv4[q2][q].z;
                  acc[4 * q + 3] += wc * pv4[q2][q].w;
                }
              }
            }
            __nv_bfloat16* dst = P.o + (static_cast<size_t>(s) * B + sl2) * nq * TD + static_cast<size_t>(hrow) * TD + d;
            uint4 hv[2], lv[2];
            __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(hv);
            __nv_bfloat162* lp = reinterpret_cast<__nv_bfloat162*>(lv);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              hp[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
              const float2 f = __bfloat1622float2(hp[q]);
              lp[q] = __floats2bfloat162_rn(acc[2 * q] - f.x, acc[2 * q + 1] - f.y);
            }
            reinterpret_cast<uint4*>(dst)[0] = hv[0];
            reinterpret_cast<uint4*>(dst)[1] = hv[1];
            reinterpret_cast<uint4*>(dst + static_cast<size_t>(P.o_lo) * nq * TD)[0] = lv[0];
            reinterpret_cast<uint4*>(dst + static_cast<size_t>(P.o_lo) * nq * TD)[1] = lv[1];
          }
          if (r == 0) tl_stamp(tl, 9);
        }
        named_bar_sync(1, TR);  // s_flag[1] and the merge tables are reused by the next segment
      }
      j += seg;
    }
    if (r == 0) tl_stamp(tl, 7);
    if (tl && r == 0) {
      tl[12] = t_ws;
      tl[13] = t_wpv;
      tl[14] = static_cast<unsigned long long>(n);
    }
  }

  // ---- every MMA has completed (the issuer waited for them) before TMEM is released
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) tl_stamp(tl, kTlExit);
}

int attn_tc_smem(int batch) { return 1024 + PRE_OFF + (batch + 1) * 4; }

int attn_tc_set_attributes() {
  return static_cast<int>(cudaFuncSetAttribute(attn_flat_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               attn_tc_smem(kTcMaxBatch)));
}

bool attn_tc_supported(const AttnParams& p) {
  return p.d == TD && p.nq == TNW * p.nkv && p.nkv % 2 == 0 && p.B <= 16 && p.batch <= kTcMaxBatch;
}

int launch_attention_flat_tc(const AttnParams& p, int n_ctas, cudaStream_t stream, bool pdl) {
  if (!attn_tc_supported(p) || p.batch < 1 || n_ctas < 1 || n_ctas > kMaxCtas)
    return static_cast<int>(cudaErrorInvalidValue);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas, 1, 1);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = attn_tc_smem(p.batch);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, attn_flat_tc_kernel, p));
}

}  // namespace dfl
