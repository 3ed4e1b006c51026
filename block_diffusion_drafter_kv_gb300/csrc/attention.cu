// Bidirectional block attention of the DFlash drafter (sm_103a).
//
// Every slot of the block attends, without a causal mask, to all injected context keys
// [0, len) and to the block's own B keys [len, len+B) (jansverre.net, "Hva gjør DFlash
// annerledes enn vanlig spekulativ dekoding?": the masked block is denoised in a single
// pass; theaistack.guide, "L'idea chiave": the injected K/V live in the draft KV cache).
// The block's keys were written into the cache at [len, len+B) by the Q/K/V epilogue, so
// the key range is one contiguous run.
//
// Split-KV flash decoding: one thread-block cluster per (sequence, KV head); the CTAs of
// the cluster split the key range. In a CTA, warp w serves query head g*group + w % group for
// all (<= 16) block slots, so the group's query heads share every K/V tile staged in shared
// memory by TMA. With two key groups (2 * group warps), warps w and w + group serve the same
// head and take alternate tiles, so each SM sub-partition has two independent MMA chains to
// interleave; their states are combined in shared memory after the key loop. QKᵀ and PV run on the tensor cores with fp16 operands (q, the fp16 K and V
// caches, the probabilities) accumulating in fp32, with an online softmax in registers. The CTAs' partial (max, sum, output) are merged through distributed shared
// memory in a fixed order, so no partials touch HBM. The output is written as a high bf16
// plane and a low plane (the bf16 of the remainder) for the output projection.
#include "attn_tile.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int KT = kAttnKeys;  // keys per tile
static_assert(KT == kPageRows, "a key tile is one page of a paged cache");
constexpr int STAGES = 3;

// Offset of the merge inputs from the 1024-aligned base: the ring of fp16 K + V tiles, its
// full/empty barriers, the merge barrier and two flags.
__host__ __device__ constexpr int attn_recv_offset(int D) {
  return (STAGES * KT * D * 4 + (2 * STAGES + 1) * 8 + 8 + 15) / 16 * 16;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(256) attn_kernel(const __grid_constant__ AttnParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_ATTN) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  constexpr int K_BYTES = KT * D * 2;  // fp16 K tile
  constexpr int V_BYTES = KT * D * 2;  // fp16 V tile
  constexpr int TILE_BYTES = K_BYTES + V_BYTES;
  constexpr int NT_D = D / 8;   // n-tiles over d in the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * TILE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* recv_bar = empty + STAGES;  // the peers' partials of the rows this CTA merges
  volatile int* s_flag = reinterpret_cast<volatile int*>(recv_bar + 1);  // [0] abort, [1] merge input ok
  float* s_stage = reinterpret_cast<float*>(smem);  // after the key loop: partials by merging CTA
  float* s_recv = reinterpret_cast<float*>(smem + attn_recv_offset(D));

  const int nw = P.nq / P.nkv;                   // warps per key group: the GQA group
  const int KW = (blockDim.x >> 5) / nw;         // key groups (1 or 2)
  const int warp = (threadIdx.x >> 5) % nw, kg = (threadIdx.x >> 5) / nw, lane = threadIdx.x & 31;
  const int g = blockIdx.y, seq = blockIdx.z;
  const int S = gridDim.x;
  const int rank = static_cast<int>(cluster_ctarank());
  const int B = P.B;
  // The cluster's CTAs merge the nw*16 query rows in slices of `per` rows: rows [k*per,
  // (k+1)*per) go to CTA k. CTA k receives from CTA c one block of partials at s_recv +
  // c*nk*(D+4): its nk rows' outputs (D floats each), then their (max, sum, 0, 0).
  const int R = nw * 16;
  const int per = (R + S - 1) / S;
  auto rows_of = [&](int k) { return max(0, min(per, R - k * per)); };
  const int nrow = rows_of(rank);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nw);
    }
    mbar_init(recv_bar, 1);
    s_flag[0] = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(S * nrow * (D + 4) * 4));
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&P.kmap);
    tma_prefetch_desc(&P.vmap);
  }
  __syncthreads();
  cluster_arrive_relaxed();  // peers may write this CTA's merge inputs once every CTA is here

  // The kernel before this one (the Q/K/V projection) starts only after the injection of
  // this step has completed, so len and the injected context keys [0, len) are final here;
  // only q and the block's own keys [len, len+B) are still being written. Tiles entirely
  // below len are therefore fetched before waiting on the previous kernel.
  const int len = __ldcg(P.len + seq);
  int nkeys = len + B;
  if (nkeys > P.cap) nkeys = P.cap;
  const int ntiles = (nkeys + KT - 1) / KT;
  const int t0 = rank * ntiles / S, t1 = (rank + 1) * ntiles / S;
  const int n = t1 - t0;
  const int key_row0 = seq * P.cap;
  const int pre = n < STAGES ? n : STAGES;

  auto issue = [&](int i, uint64_t pol) {
    const int st = i % STAGES;
    uint8_t* kd = smem + st * TILE_BYTES;
    uint8_t* vd = kd + K_BYTES;
    int row = key_row0 + (t0 + i) * KT;
    if (P.page_table) {  // tile t of a sequence is its page t
      const int page = __ldcg(P.page_table + static_cast<size_t>(seq) * P.pages_per_seq + t0 + i);
      if (page < 0 || page >= P.n_pages) raise_flag(P.err, kDevCapacity);
      row = (page < 0 || page >= P.n_pages) ? 0 : page * KT;
    }
    mbar_arrive_expect_tx(&full[st], TILE_BYTES);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_3d(kd + b * KT * 128, &P.kmap, &full[st], b * 64, g, row, pol);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_3d(vd + b * KT * 128, &P.vmap, &full[st], b * 64, g, row, pol);
  };
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_last();
    for (int i = 0; i < pre; ++i)
      if ((t0 + i + 1) * KT <= len) issue(i, pol);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) tl_stamp(tl, 5);
  if (threadIdx.x == 0) {
    const uint64_t pol = policy_evict_last();
    for (int i = 0; i < pre; ++i)
      if ((t0 + i + 1) * KT > len) issue(i, pol);
  }
  int issued = pre;  // thread 0: tiles issued so far (in order)

  // Q fragments of this warp's head: rows = block slots (>= B are zero).
  const int nq = P.nq;
  const int h = g * nw + warp;
  const int r0 = lane >> 2, kq = (lane & 3) * 2;
  FaState<D> fa;
  fa_begin<D>(fa, P.q, static_cast<size_t>(seq) * B, static_cast<size_t>(nq) * D, h, B, lane);

  for (int i = kg; i < n; i += KW) {
    const int st = i % STAGES;
    if (!s_flag[0] && !mbar_wait(&full[st], (i / STAGES) & 1, P.wait_ns)) {
      s_flag[0] = 1;
      raise_flag(P.err, kDevTimeout);
    }
    if (i == 0 && threadIdx.x == 0) tl_stamp(tl, 6);
    const uint32_t kb = smem_u32(smem + st * TILE_BYTES);
    fa_tile<D>(fa, kb, kb + K_BYTES, (t0 + i) * KT, nkeys, P.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    // Thread 0 refills the ring in tile order: every tile up to the other key group's next
    // one plus the ring depth. Tile j reuses the stage of tile j - STAGES, consumed either
    // by this warp (tile i) or by the other key group (tile i + 1, already issued), so
    // the wait always ends.
    if (threadIdx.x == 0) {
      while (issued < n && issued <= i + KW + STAGES - 1 && !s_flag[0]) {
        const int sj = issued % STAGES;
        if (!mbar_wait(&empty[sj], ((issued / STAGES) - 1) & 1, P.wait_ns)) {
          s_flag[0] = 1;
          raise_flag(P.err, kDevTimeout);
          break;
        }
        issue(issued, policy_evict_last());
        ++issued;
      }
    }
  }

  if (threadIdx.x == 0) tl_stamp(tl, 7);
  fa_end<D>(fa);
  __syncthreads();  // the ring is free: every issued tile was consumed
  if (KW > 1) {
    // the second key group hands its (output, max, sum) to the first through the free ring;
    // the first rescales both to the larger max and adds them
    float4* s_o = reinterpret_cast<float4*>(smem);
    float4* s_ml = s_o + nw * NT_D * 32;
    if (kg == 1) {
#pragma unroll
      for (int nt = 0; nt < NT_D; ++nt)
        s_o[(warp * NT_D + nt) * 32 + lane] = make_float4(fa.o[nt][0], fa.o[nt][1], fa.o[nt][2], fa.o[nt][3]);
      s_ml[warp * 32 + lane] = make_float4(fa.m[0], fa.m[1], fa.l[0], fa.l[1]);
    }
    __syncthreads();
    if (kg == 0) {
      const float4 ml = s_ml[warp * 32 + lane];
      const float mb[2] = {ml.x, ml.y}, lb[2] = {ml.z, ml.w};
      float ca[2], cb[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float M = fmaxf(fa.m[r], mb[r]);
        ca[r] = fa.m[r] == -INFINITY ? 0.f : exp2f(fa.m[r] - M);
        cb[r] = mb[r] == -INFINITY ? 0.f : exp2f(mb[r] - M);
        fa.l[r] = fa.l[r] * ca[r] + lb[r] * cb[r];
        fa.m[r] = M;
      }
#pragma unroll
      for (int nt = 0; nt < NT_D; ++nt) {
        const float4 ob = s_o[(warp * NT_D + nt) * 32 + lane];
        fa.o[nt][0] = fa.o[nt][0] * ca[0] + ob.x * cb[0];
        fa.o[nt][1] = fa.o[nt][1] * ca[0] + ob.y * cb[0];
        fa.o[nt][2] = fa.o[nt][2] * ca[1] + ob.z * cb[1];
        fa.o[nt][3] = fa.o[nt][3] * ca[1] + ob.w * cb[1];
      }
    }
    __syncthreads();
  }
  if (kg == 0) {
    // stage this CTA's partial output and (max, sum) of every row in the ring, in one block
    // per merging CTA k: [rows of k: D floats each][rows of k: (max, sum, 0, 0)]
    const int ra = warp * 16 + r0, rb = ra + 8;
    auto stage_row = [&](int rr, int hi) {
      const int k = rr / per, lr = rr - k * per;
      float* blk = s_stage + static_cast<size_t>(k) * per * (D + 4);
#pragma unroll
      for (int nt = 0; nt < NT_D; ++nt)
        *reinterpret_cast<float2*>(blk + lr * D + nt * 8 + kq) = make_float2(fa.o[nt][2 * hi], fa.o[nt][2 * hi + 1]);
      if ((lane & 3) == 0)
        *reinterpret_cast<float4*>(blk + rows_of(k) * D + lr * 4) = make_float4(fa.m[hi], fa.l[hi], 0.f, 0.f);
    };
    stage_row(ra, 0);
    stage_row(rb, 1);
  }
  fence_async_shared();  // the bulk copies below read the staged partials
  __syncthreads();
  cluster_wait();  // every CTA of the cluster has started and armed its merge barrier
  if (threadIdx.x < 32 && lane < S) {  // one bulk copy per merging CTA, each from its own lane
    const int k = lane, nk = rows_of(k);
    if (nk > 0) {
      const uint32_t bytes = static_cast<uint32_t>(nk * (D + 4) * 4);
      const uint32_t src = smem_u32(s_stage) + static_cast<uint32_t>(k * per * (D + 4) * 4);
      const uint32_t dst = smem_u32(s_recv) + static_cast<uint32_t>(rank * nk * (D + 4) * 4);
      bulk_copy_to_peer(map_shared_rank(dst, k), src, bytes, map_shared_rank(smem_u32(recv_bar), k));
    }
    bulk_commit();
  }
  if (threadIdx.x == 0) tl_stamp(tl, 8);

  // merge the rows [rank*per, rank*per + nrow): block c of s_recv came from CTA c
  if (nrow > 0) {
    if (threadIdx.x == 0) {
      const bool ok = mbar_wait(recv_bar, 0, P.wait_ns);
      if (!ok) raise_flag(P.err, kDevTimeout);
      s_flag[1] = ok ? 1 : 0;
    }
    __syncthreads();
    if (s_flag[1]) {
      const int blk = nrow * (D + 4);
      const int items = nrow * (D / 4);
      for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int lr = it / (D / 4), d = (it % (D / 4)) * 4;
        const int rr = rank * per + lr;
        const int w = rr >> 4, slot = rr & 15;
        if (slot >= B) continue;
        // split weights exp2(m_c - M) / sum_c' exp2(m_c' - M) l_c', combined in CTA order
        const float* ml = s_recv + nrow * D + lr * 4;
        float M = -INFINITY;
        for (int c = 0; c < S; ++c) M = fmaxf(M, ml[c * blk]);
        float den = 0.f;
        for (int c = 0; c < S; ++c) {
          const float mc = ml[c * blk];
          den += (mc == -INFINITY ? 0.f : exp2f(mc - M)) * ml[c * blk + 1];
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < S; ++c) {
          const float mc = ml[c * blk];
          const float wt = (mc == -INFINITY ? 0.f : exp2f(mc - M)) * inv;
          const float4 part = *reinterpret_cast<const float4*>(s_recv + c * blk + lr * D + d);
          acc.x += wt * part.x;
          acc.y += wt * part.y;
          acc.z += wt * part.z;
          acc.w += wt * part.w;
        }
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(acc.x, acc.y), h23 = __floats2bfloat162_rn(acc.z, acc.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(acc.x - f01.x, acc.y - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(acc.z - f23.x, acc.w - f23.y);
        uint2 ph, pl;
        ph.x = *reinterpret_cast<const uint32_t*>(&h01);
        ph.y = *reinterpret_cast<const uint32_t*>(&h23);
        pl.x = *reinterpret_cast<const uint32_t*>(&l01);
        pl.y = *reinterpret_cast<const uint32_t*>(&l23);
        __nv_bfloat16* dst =
            P.o + (static_cast<size_t>(seq) * B + slot) * nq * D + static_cast<size_t>(g * nw + w) * D + d;
        *reinterpret_cast<uint2*>(dst) = ph;
        *reinterpret_cast<uint2*>(dst + static_cast<size_t>(P.o_lo) * nq * D) = pl;
      }
    }
  }
  if (threadIdx.x == 0) tl_stamp(tl, 9);
  // the staged partials stay in place until the peers' copies have read them; every copy
  // into this CTA's memory has landed (its merge barrier completed) or this CTA merges none
  if (threadIdx.x < 32 && lane < S) bulk_wait_read();
  if (threadIdx.x == 0) tl_stamp(tl, kTlExit);
}

// ---------------------------------------------------------------------------------------
// Key-split attention over one flat tile list, for ragged or large batches.
//
// The key tiles of every (sequence, KV head) pair, pairs in (sequence, head) order, form one
// list of T tiles cut into G equal contiguous ranges, one per CTA (one CTA per SM): every SM
// gets the same number of tiles whatever the lengths. A CTA walks its range as segments,
// one per pair it touches. A pair that lies inside one range is normalised and written by
// its CTA. A pair cut between CTAs is merged by the last of them to finish (an arrival
// counter per pair): each writes its unnormalised output and per-row (max, sum) to a slot,
// 2c for CTA c's first segment and 2c + 1 for its last, and the last to arrive combines the
// slots in CTA order, so the result does not depend on the order of arrival.
constexpr int FST = 3;                                    // ring depth of the flat kernel
constexpr int kFlatHdr = (2 * FST * 8 + 16 + 15) / 16 * 16;  // its full/empty barriers and flags
__host__ __device__ constexpr int attn_flat_fixed_smem(int D, int nw) {
  // 1024 alignment slack, the ring, barriers and flags, the second key group's output and
  // (max, sum) for the combine, the merge's row statistics and contributor slots
  return 1024 + FST * KT * D * 4 + kFlatHdr + nw * (D / 8) * 32 * 16 + nw * 32 * 16 + 2 * 128 * 4 + kMaxCtas * 4;
}

DEV long long flat_begin(int c, long long T, int G) { return static_cast<long long>(c) * T / G; }
// CTA whose range holds flat tile u.
DEV int flat_cta_of(long long u, long long T, int G) {
  return static_cast<int>(((u + 1) * G + T - 1) / T) - 1;
}

template <int D>
__global__ void __launch_bounds__(256) attn_flat_kernel(const __grid_constant__ AttnParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>(blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_ATTN) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  constexpr int K_BYTES = KT * D * 2;
  constexpr int TILE_BYTES = 2 * K_BYTES;
  constexpr int NT_D = D / 8;
  const int nw = P.nq / P.nkv;                // warps per key group: the GQA group
  const int KW = (blockDim.x >> 5) / nw;      // key groups (1 or 2)
  const int warp = (threadIdx.x >> 5) % nw, kg = (threadIdx.x >> 5) / nw, lane = threadIdx.x & 31;
  const int r0 = lane >> 2, kq = (lane & 3) * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + FST * TILE_BYTES);
  uint64_t* empty = full + FST;
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + FST * TILE_BYTES + 2 * FST * 8);  // [0] abort, [1] last
  float4* s_o = reinterpret_cast<float4*>(smem + FST * TILE_BYTES + kFlatHdr);
  float4* s_ml = s_o + nw * NT_D * 32;
  float* s_rm = reinterpret_cast<float*>(s_ml + nw * 32);  // merge: each row's max
  float* s_rinv = s_rm + 128;                               // and 1 / normaliser
  int* s_cs = reinterpret_cast<int*>(s_rinv + 128);         // merge: contributor slots, [G]
  int* s_pre = s_cs + kMaxCtas;                             // [batch + 1]: tiles per head before sequence s

  const int batch = P.batch, B = P.B, nkv = P.nkv, nq = P.nq;
  // The kernel before this one (the Q/K/V projection) starts only after the injection of
  // this step has completed, so len and the injected context keys [0, len) are final here.
  for (int s = threadIdx.x; s < batch; s += blockDim.x) {
    int nk = __ldcg(P.len + s) + B;
    if (nk > P.cap) nk = P.cap;
    s_pre[s + 1] = (nk + KT - 1) / KT;
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < FST; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], nw);
    }
    s_flag[0] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&P.kmap);
    tma_prefetch_desc(&P.vmap);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s_pre[0] = 0;
    for (int s = 0; s < batch; ++s) s_pre[s + 1] += s_pre[s];
  }
  __syncthreads();

  const long long T = static_cast<long long>(nkv) * s_pre[batch];
  const int G = gridDim.x, c = blockIdx.x;
  const long long T0 = flat_begin(c, T, G);
  const int n = static_cast<int>(flat_begin(c + 1, T, G) - T0);
  // flat tile u -> sequence s, head g, tile t of the pair, the pair's tile count nt
  auto locate = [&](long long u, int& s, int& g, int& t, int& nt) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(nkv) * s_pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
    nt = s_pre[s + 1] - s_pre[s];
    const long long r = u - static_cast<long long>(nkv) * s_pre[s];
    g = static_cast<int>(r / nt);
    t = static_cast<int>(r - static_cast<long long>(g) * nt);
  };
  auto issue_at = [&](int j, int s, int g, int t, uint64_t pol) {
    const int st = j % FST;
    uint8_t* kd = smem + st * TILE_BYTES;
    uint8_t* vd = kd + K_BYTES;
    int row = s * P.cap + t * KT;
    if (P.page_table) {  // tile t of a sequence is its page t
      const int page = __ldcg(P.page_table + static_cast<size_t>(s) * P.pages_per_seq + t);
      if (page < 0 || page >= P.n_pages) raise_flag(P.err, kDevCapacity);
      row = (page < 0 || page >= P.n_pages) ? 0 : page * KT;
    }
    mbar_arrive_expect_tx(&full[st], TILE_BYTES);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_3d(kd + b * KT * 128, &P.kmap, &full[st], b * 64, g, row, pol);
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_3d(vd + b * KT * 128, &P.vmap, &full[st], b * 64, g, row, pol);
  };
  // K/V read once per call: streamed through L2 unless the layer's cache is small enough to
  // stay there until the next step (16 MB, one eighth of L2, per layer)
  const uint64_t kv_pol = T * TILE_BYTES > (16ll << 20) ? policy_evict_first() : policy_evict_last();
  const int pre = n < FST ? n : FST;
  // tiles entirely below len do not depend on the previous kernel: fetched before waiting
  auto below_len = [&](int j) {
    int s, g, t, nt;
    locate(T0 + j, s, g, t, nt);
    return (t + 1) * KT <= __ldcg(P.len + s);
  };
  auto issue = [&](int j, uint64_t pol) {
    int s, g, t, nt;
    locate(T0 + j, s, g, t, nt);
    issue_at(j, s, g, t, pol);
  };
  if (threadIdx.x == 0) {
    const uint64_t pol = kv_pol;
    for (int j = 0; j < pre; ++j)
      if (below_len(j)) issue(j, pol);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    tl_stamp(tl, 5);
    const uint64_t pol = kv_pol;
    for (int j = 0; j < pre; ++j)
      if (!below_len(j)) issue(j, pol);
  }
  int issued = pre;  // thread 0: tiles issued so far (in order)
  // thread 0: (sequence, head, tile, tiles of the pair) of tile `issued`, advanced in order
  int cs = 0, cg = 0, ct = 0, cnt = 1;
  if (threadIdx.x == 0 && issued < n) locate(T0 + issued, cs, cg, ct, cnt);
  // Thread 0 refills the ring in order up to tile `upto`, waiting only for stages whose
  // previous tile lies before `bound`: tiles the CTA consumes before its next CTA-wide
  // barrier, so that every wait ends.
  auto refill = [&](int upto, int bound) {
    while (issued < n && issued <= upto && issued - FST < bound && !s_flag[0]) {
      const int sj = issued % FST;
      if (issued >= FST && !mbar_wait(&empty[sj], ((issued / FST) - 1) & 1, P.wait_ns)) {
        s_flag[0] = 1;
        raise_flag(P.err, kDevTimeout);
        break;
      }
      issue_at(issued, cs, cg, ct, kv_pol);
      ++issued;
      if (++ct == cnt) {
        ct = 0;
        if (++cg == nkv) {
          cg = 0;
          ++cs;
          if (cs < batch) cnt = s_pre[cs + 1] - s_pre[cs];
        }
      }
    }
  };

  const size_t slot_floats = static_cast<size_t>(nw) * 16 * (D + 4);
  bool merged = false;  // thread 0: timeline stamp of the first merge
  for (int j = 0; j < n;) {
    int s, g, ta, nt;
    locate(T0 + j, s, g, ta, nt);
    const int seg = min(n - j, nt - ta);
    const bool whole = ta == 0 && seg == nt;
    int nkeys = __ldcg(P.len + s) + B;
    if (nkeys > P.cap) nkeys = P.cap;
    if (threadIdx.x == 0) refill(j + KW + FST - 1, j);
    const int h = g * nw + warp;
    FaState<D> fa;
    fa_begin<D>(fa, P.q, static_cast<size_t>(s) * B, static_cast<size_t>(nq) * D, h, B, lane);
    for (int i = j + ((kg - j % KW) + KW) % KW; i < j + seg; i += KW) {
      const int st = i % FST;
      if (!s_flag[0] && !mbar_wait(&full[st], (i / FST) & 1, P.wait_ns)) {
        s_flag[0] = 1;
        raise_flag(P.err, kDevTimeout);
      }
      if (i == 0 && threadIdx.x == 0) tl_stamp(tl, 6);
      const uint32_t kb = smem_u32(smem + st * TILE_BYTES);
      fa_tile<D>(fa, kb, kb + K_BYTES, (ta + i - j) * KT, nkeys, P.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (threadIdx.x == 0) refill(i + KW + FST - 1, j + seg);
    }
    fa_end<D>(fa);
    if (KW > 1) {
      // the second key group hands its (output, max, sum) to the first, which rescales both
      // to the larger max and adds them
      if (kg == 1) {
#pragma unroll
        for (int nt2 = 0; nt2 < NT_D; ++nt2)
          s_o[(warp * NT_D + nt2) * 32 + lane] = make_float4(fa.o[nt2][0], fa.o[nt2][1], fa.o[nt2][2], fa.o[nt2][3]);
        s_ml[warp * 32 + lane] = make_float4(fa.m[0], fa.m[1], fa.l[0], fa.l[1]);
      }
      __syncthreads();
      if (kg == 0) {
        const float4 ml = s_ml[warp * 32 + lane];
        const float mb[2] = {ml.x, ml.y}, lb[2] = {ml.z, ml.w};
        float ca[2], cb[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float M = fmaxf(fa.m[r], mb[r]);
          ca[r] = fa.m[r] == -INFINITY ? 0.f : exp2f(fa.m[r] - M);
          cb[r] = mb[r] == -INFINITY ? 0.f : exp2f(mb[r] - M);
          fa.l[r] = fa.l[r] * ca[r] + lb[r] * cb[r];
          fa.m[r] = M;
        }
#pragma unroll
        for (int nt2 = 0; nt2 < NT_D; ++nt2) {
          const float4 ob = s_o[(warp * NT_D + nt2) * 32 + lane];
          fa.o[nt2][0] = fa.o[nt2][0] * ca[0] + ob.x * cb[0];
          fa.o[nt2][1] = fa.o[nt2][1] * ca[0] + ob.y * cb[0];
          fa.o[nt2][2] = fa.o[nt2][2] * ca[1] + ob.z * cb[1];
          fa.o[nt2][3] = fa.o[nt2][3] * ca[1] + ob.w * cb[1];
        }
      }
    }
    if (whole) {
      // the pair lies in this CTA's range: normalise and write both bf16 planes
      if (kg == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int slot = r0 + 8 * hr;
          if (slot >= B) continue;
          const float inv = fa.l[hr] > 0.f ? 1.f / fa.l[hr] : 0.f;
          __nv_bfloat16* dst = P.o + (static_cast<size_t>(s) * B + slot) * nq * D + static_cast<size_t>(h) * D;
#pragma unroll
          for (int nt2 = 0; nt2 < NT_D; ++nt2) {
            const float v0 = fa.o[nt2][2 * hr] * inv, v1 = fa.o[nt2][2 * hr + 1] * inv;
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v0, v1);
            const float2 hf = __bfloat1622float2(hi);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
            *reinterpret_cast<__nv_bfloat162*>(dst + nt2 * 8 + kq) = hi;
            *reinterpret_cast<__nv_bfloat162*>(dst + static_cast<size_t>(P.o_lo) * nq * D + nt2 * 8 + kq) = lo;
          }
        }
      }
    } else {
      // a cut pair: this CTA's part to its slot, then count it in
      const long long base = static_cast<long long>(nkv) * s_pre[s] + static_cast<long long>(g) * nt;
      float* slot_p = P.part + (2 * static_cast<size_t>(c) + (j == 0 ? 0 : 1)) * slot_floats;
      if (kg == 0) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int rr = warp * 16 + r0 + 8 * hr;
          if (r0 + 8 * hr >= B) continue;
#pragma unroll
          for (int nt2 = 0; nt2 < NT_D; ++nt2)
            __stcg(reinterpret_cast<float2*>(slot_p + static_cast<size_t>(rr) * D + nt2 * 8 + kq),
                   make_float2(fa.o[nt2][2 * hr], fa.o[nt2][2 * hr + 1]));
          if ((lane & 3) == 0)
            __stcg(reinterpret_cast<float4*>(slot_p + static_cast<size_t>(nw) * 16 * D + rr * 4),
                   make_float4(fa.m[hr], fa.l[hr], 0.f, 0.f));
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        const int c_first = flat_cta_of(base, T, G), c_last = flat_cta_of(base + nt - 1, T, G);
        int n_c = 0;  // CTAs with a part of the pair (CTAs with an empty range have none)
        for (int cc = c_first; cc <= c_last; ++cc) n_c += flat_begin(cc + 1, T, G) > flat_begin(cc, T, G);
        __threadfence();
        const int old = atomicAdd(P.cnt + s * nkv + g, 1);
        const int last = old == n_c - 1;
        if (last) {
          P.cnt[s * nkv + g] = 0;
          __threadfence();
        }
        s_flag[1] = last;
      }
      __syncthreads();
      if (s_flag[1]) {
        if (threadIdx.x == 0 && !merged) tl_stamp(tl, 8);
        merged = true;
        // Combine the parts in CTA order: out = sum_c exp2(m_c - M) o_c / sum_c exp2(m_c - M) l_c.
        // The contributors' slots first, then each row's max and normaliser, then the rows in
        // 16-float blocks with every contributor's loads of a block in flight together.
        const int c_first = flat_cta_of(base, T, G), c_last = flat_cta_of(base + nt - 1, T, G);
        const int nk = c_last - c_first + 1;
        const int R = nw * 16;
        for (int k = threadIdx.x; k < nk; k += blockDim.x) {
          const int cc = c_first + k;
          const long long b0 = flat_begin(cc, T, G);
          s_cs[k] = flat_begin(cc + 1, T, G) > b0 ? 2 * cc + (b0 >= base ? 0 : 1) : -1;
        }
        __syncthreads();
        for (int rr = threadIdx.x; rr < R; rr += blockDim.x) {
          if ((rr & 15) >= B) continue;
          float M = -INFINITY, den = 0.f;
#pragma unroll 4
          for (int k = 0; k < nk; ++k) {
            const int sl = s_cs[k];
            if (sl < 0) continue;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(P.part + sl * slot_floats + static_cast<size_t>(R) * D + rr * 4));
            if (ml.x == -INFINITY) continue;
            if (ml.x > M) {
              den = den * exp2f(M - ml.x) + ml.y;
              M = ml.x;
            } else {
              den += ml.y * exp2f(ml.x - M);
            }
          }
          s_rm[rr] = M;
          s_rinv[rr] = den > 0.f ? 1.f / den : 0.f;
        }
        __syncthreads();
        for (int it = threadIdx.x; it < R * (D / 16); it += blockDim.x) {
          const int rr = it / (D / 16), d = (it % (D / 16)) * 16;
          const int w = rr >> 4, slot = rr & 15;
          if (slot >= B) continue;
          const float M = s_rm[rr], inv = s_rinv[rr];
          float acc[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) acc[q] = 0.f;
#pragma unroll 2
          for (int k = 0; k < nk; ++k) {
            const int sl = s_cs[k];
            if (sl < 0) continue;
            const float* sp = P.part + sl * slot_floats;
            const float mc = __ldcg(sp + static_cast<size_t>(R) * D + rr * 4);
            float4 pv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) pv[q] = __ldcg(reinterpret_cast<const float4*>(sp + static_cast<size_t>(rr) * D + d + 4 * q));
            const float wc = mc == -INFINITY ? 0.f : exp2f(mc - M) * inv;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[4 * q] += wc * pv[q].x;
              acc[4 * q + 1] += wc * pv[q].y;
              acc[4 * q + 2] += wc * pv[q].z;
              acc[4 * q + 3] += wc * pv[q].w;
            }
          }
          __nv_bfloat16* dst =
              P.o + (static_cast<size_t>(s) * B + slot) * nq * D + static_cast<size_t>(g * nw + w) * D + d;
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
          reinterpret_cast<uint4*>(dst + static_cast<size_t>(P.o_lo) * nq * D)[0] = lv[0];
          reinterpret_cast<uint4*>(dst + static_cast<size_t>(P.o_lo) * nq * D)[1] = lv[1];
        }
        if (threadIdx.x == 0) tl_stamp(tl, 9);
      }
    }
    __syncthreads();  // the combine buffers and s_flag[1] are reused by the next segment
    j += seg;
  }
  if (threadIdx.x == 0) {
    tl_stamp(tl, 7);
    // after an abandoned wait, the copies still in flight land before the CTA exits
    if (s_flag[0])
      for (int q = issued > FST ? issued - FST : 0; q < issued; ++q)
        if (!mbar_wait(&full[q % FST], (q / FST) & 1, P.wait_ns)) break;
    tl_stamp(tl, kTlExit);
  }
}

// Dynamic shared memory: the tile ring (which holds this CTA's staged partials after the
// key loop), its barriers, and the merge inputs from every CTA of the cluster.
static int attn_smem(int D, int nw, int split) {
  const int R = nw * 16, per = (R + split - 1) / split;
  return 1024 + attn_recv_offset(D) + split * per * (D + 4) * 4;
}
static int attn_smem_max(int D) { return attn_smem(D, 8, 16); }

int attn_flat_smem(int D, int nw, int batch) { return attn_flat_fixed_smem(D, nw) + (batch + 1) * 4; }

int attn_set_attributes() {
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_flat_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_flat_smem(128, 4, kAttnFlatMaxBatch));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_flat_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_flat_smem(64, 8, kAttnFlatMaxBatch));
#define DFL_ATTN_ATTR(D)                                                                                   \
  if (e == cudaSuccess)                                                                                    \
    e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem_max(D)); \
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  DFL_ATTN_ATTR(64) DFL_ATTN_ATTR(128)
#undef DFL_ATTN_ATTR
  return static_cast<int>(e);
}

// How many clusters of `split` CTAs of the head-dim-128 kernel the device can hold at once
// (clusters above 8 CTAs need that many free SMs in one GPC); 0 if it cannot run one.
int attn_resident_clusters(int split) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, 1, 1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = attn_smem_max(128);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<128>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

template <int D>
static int launch_d(const AttnParams& p, int batch, int split, cudaStream_t stream, bool pdl) {
  const int group = p.nq / p.nkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, p.nkv, batch);
  cfg.blockDim = dim3(32 * group * p.key_groups);
  cfg.dynamicSmemBytes = attn_smem(D, group, split);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, attn_kernel<D>, p));
}

template <int D>
static int launch_flat_d(const AttnParams& p, int n_ctas, cudaStream_t stream, bool pdl) {
  const int group = p.nq / p.nkv;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas, 1, 1);
  cfg.blockDim = dim3(32 * group * p.key_groups);
  cfg.dynamicSmemBytes = attn_flat_smem(D, group, p.batch);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, attn_flat_kernel<D>, p));
}

int launch_attention_flat(const AttnParams& p, int n_ctas, cudaStream_t stream, bool pdl) {
  if (p.batch < 1 || p.batch > kAttnFlatMaxBatch || n_ctas < 1 || n_ctas > kMaxCtas) return static_cast<int>(cudaErrorInvalidValue);
  if (p.d == 128) return launch_flat_d<128>(p, n_ctas, stream, pdl);
  if (p.d == 64) return launch_flat_d<64>(p, n_ctas, stream, pdl);
  return static_cast<int>(cudaErrorInvalidValue);
}

int launch_attention(const AttnParams& p, int batch, int split, cudaStream_t stream, bool pdl) {
  if (p.d == 128) return launch_d<128>(p, batch, split, stream, pdl);
  if (p.d == 64) return launch_d<64>(p, batch, split, stream, pdl);
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace dfl
