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
// the cluster split the key range. In a CTA, warp w serves query head g*group + w for all
// (<= 16) block slots, so the group's query heads share every K/V tile staged in shared
// memory by TMA. QKᵀ runs on the tensor cores in TF32 against the fp32 K cache and PV in
// bf16 against the bf16 V cache, both accumulating in fp32, with an online softmax in
// registers. The CTAs' partial (max, sum, output) are merged through distributed shared
// memory in a fixed order, so no partials touch HBM. The output is written as a high bf16
// plane and a low plane (the bf16 of the remainder) for the output projection.
#include "attn_tile.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int KT = kAttnKeys;  // keys per tile
constexpr int STAGES = 3;

}  // namespace

template <int D>
__global__ void __launch_bounds__(256) attn_kernel(const __grid_constant__ AttnParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_ATTN) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  constexpr int K_BYTES = KT * D * 4;  // fp32 K tile
  constexpr int V_BYTES = KT * D * 2;  // bf16 V tile
  constexpr int TILE_BYTES = K_BYTES + V_BYTES;
  constexpr int NT_D = D / 8;   // n-tiles over d in the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * TILE_BYTES);
  uint64_t* empty = full + STAGES;
  float* s_m = reinterpret_cast<float*>(empty + STAGES);  // [128] per-row running max (log2 units)
  float* s_l = s_m + 128;                                  // [128] per-row sum
  float* s_w = s_l + 128;                                  // [128 rows][16] combine weights
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_w + 128 * 16);
  float* s_o = reinterpret_cast<float*>(smem);             // [rows][D] after the key loop

  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y, seq = blockIdx.z;
  const int S = gridDim.x;
  const int rank = static_cast<int>(cluster_ctarank());
  const int B = P.B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nw);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&P.kmap);
    tma_prefetch_desc(&P.vmap);
  }
  __syncthreads();

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
    const int row = key_row0 + (t0 + i) * KT;
    mbar_arrive_expect_tx(&full[st], TILE_BYTES);
#pragma unroll
    for (int b = 0; b < D / 32; ++b) tma_load_3d(kd + b * KT * 128, &P.kmap, &full[st], b * 32, g, row, pol);
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

  // Q fragments of this warp's head: rows = block slots (>= B are zero).
  const int nq = P.nq;
  const int h = g * nw + warp;
  const int r0 = lane >> 2, kq = (lane & 3) * 2;
  FaState<D> fa;
  fa_begin<D>(fa, P.q, static_cast<size_t>(seq) * B, static_cast<size_t>(nq) * D, h, B, lane);

  for (int i = 0; i < n; ++i) {
    const int st = i % STAGES;
    if (!*s_abort && !mbar_wait(&full[st], (i / STAGES) & 1)) {
      *s_abort = 1;
      raise_flag(P.err, kDevTimeout);
    }
    if (i == 0 && threadIdx.x == 0) tl_stamp(tl, 6);
    const uint32_t kb = smem_u32(smem + st * TILE_BYTES);
    fa_tile<D>(fa, kb, kb + K_BYTES, (t0 + i) * KT, nkeys, P.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (threadIdx.x == 0 && i + STAGES < n) {
      if (!*s_abort && !mbar_wait(&empty[st], (i / STAGES) & 1)) {
        *s_abort = 1;
        raise_flag(P.err, kDevTimeout);
      }
      if (!*s_abort) issue(i + STAGES, policy_evict_last());
    }
  }

  if (threadIdx.x == 0) tl_stamp(tl, 7);
  fa_end<D>(fa);
  __syncthreads();  // the ring is free: every issued tile was consumed
  {
    const int ra = warp * 16 + r0, rb = ra + 8;
#pragma unroll
    for (int nt = 0; nt < NT_D; ++nt) {
      const int d = nt * 8 + kq;
      s_o[ra * D + d] = fa.o[nt][0];
      s_o[ra * D + d + 1] = fa.o[nt][1];
      s_o[rb * D + d] = fa.o[nt][2];
      s_o[rb * D + d + 1] = fa.o[nt][3];
    }
    if ((lane & 3) == 0) {
      s_m[ra] = fa.m[0];
      s_m[rb] = fa.m[1];
      s_l[ra] = fa.l[0];
      s_l[rb] = fa.l[1];
    }
  }
  cluster_sync();

  if (threadIdx.x == 0) tl_stamp(tl, 8);
  // merge: this CTA owns rows [rb0, rb1) of the nw*16 query rows. First every (row, split)
  // pair's max and sum are fetched in parallel, then each row's split weights are formed.
  const int R = nw * 16;
  const int per = (R + S - 1) / S;
  const int rb0 = rank * per, rb1 = min(R, rb0 + per);
  const int nrow = max(rb1 - rb0, 0);
  float* s_wm = s_w;              // [rows][S] remote maxima, then weights (rows*S <= 144)
  float* s_wl = s_w + 1024;       // [rows][S] remote sums
  for (int k = threadIdx.x; k < nrow * S; k += blockDim.x) {
    const int rr = rb0 + k / S, c = k % S;
    s_wm[(rr - rb0) * S + c] = ld_shared_cluster_f32(map_shared_rank(smem_u32(&s_m[rr]), c));
    s_wl[(rr - rb0) * S + c] = ld_shared_cluster_f32(map_shared_rank(smem_u32(&s_l[rr]), c));
  }
  __syncthreads();
  for (int k = threadIdx.x; k < nrow; k += blockDim.x) {
    float M = -INFINITY;
    for (int c = 0; c < S; ++c) M = fmaxf(M, s_wm[k * S + c]);
    float den = 0.f;
    for (int c = 0; c < S; ++c) {
      const float mc = s_wm[k * S + c];
      const float w = mc == -INFINITY ? 0.f : exp2f(mc - M);
      s_wm[k * S + c] = w;
      den += w * s_wl[k * S + c];
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int c = 0; c < S; ++c) s_wm[k * S + c] *= inv;
  }
  __syncthreads();
  // combine: a thread takes 4 consecutive d of one row and reads all splits' values at once
  constexpr int kMaxSplit = 16;
  const int items = nrow * (D / 4);
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int rr = rb0 + it / (D / 4), d = (it % (D / 4)) * 4;
    const int w = rr >> 4, slot = rr & 15;
    if (slot >= B) continue;
    float4 part[kMaxSplit];
    const uint32_t a = smem_u32(&s_o[rr * D + d]);
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c)
      if (c < S) part[c] = ld_shared_cluster_v4(map_shared_rank(a, c));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxSplit; ++c)
      if (c < S) {
        const float wt = s_wm[(rr - rb0) * S + c];
        acc.x += wt * part[c].x;
        acc.y += wt * part[c].y;
        acc.z += wt * part[c].z;
        acc.w += wt * part[c].w;
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
    __nv_bfloat16* dst = P.o + (static_cast<size_t>(seq) * B + slot) * nq * D + static_cast<size_t>(g * nw + w) * D + d;
    *reinterpret_cast<uint2*>(dst) = ph;
    *reinterpret_cast<uint2*>(dst + static_cast<size_t>(P.o_lo) * nq * D) = pl;
  }
  if (threadIdx.x == 0) tl_stamp(tl, 9);
  if (threadIdx.x == 0) tl_stamp(tl, kTlExit);
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
}

template <int D>
static int attn_smem() {
  return 1024 + STAGES * (KT * D * 6) + STAGES * 16 + (128 * 2 + 128 * 16) * 4 + 16;
}

int attn_set_attributes() {
  cudaError_t e = cudaSuccess;
#define DFL_ATTN_ATTR(D)                                                                                   \
  if (e == cudaSuccess)                                                                                    \
    e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem<D>()); \
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
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = attn_smem<128>();
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
  cfg.blockDim = dim3(32 * group);
  cfg.dynamicSmemBytes = attn_smem<D>();
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

int launch_attention(const AttnParams& p, int batch, int split, cudaStream_t stream, bool pdl) {
  if (p.d == 128) return launch_d<128>(p, batch, split, stream, pdl);
  if (p.d == 64) return launch_d<64>(p, batch, split, stream, pdl);
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace dfl
