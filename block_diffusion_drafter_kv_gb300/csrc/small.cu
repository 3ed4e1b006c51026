// Block initialisation, greedy verification and the synthetic-target harness kernels.
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

// ---------------------------------------------------------------- block initialisation
// Slot 0 of each sequence holds the last accepted token's embedding, slots 1..B-1 the
// mask embedding (jansverre.net, "Hva gjør DFlash annerledes ...": the drafter denoises a
// masked token block). Writes the fp32 residual x, its bf16 copy scaled by layer 0's
// attention-norm gain (the next projection's operand) and each row's sum of squares.
// All loads of a thread are issued before any of its stores (the buffers could alias as far
// as the compiler knows), so the kernel costs one memory round trip, not one per element.
__global__ void __launch_bounds__(256) embed_kernel(const EmbedParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>(blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_EMBED) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) tl_stamp(tl, 5);
  constexpr int kMaxIter = 4;  // H <= 4 * 8 * blockDim
  const int row = blockIdx.x;
  const int s = row / P.B, i = row - s * P.B;
  const __nv_bfloat16* src = P.mask_emb;
  if (i == 0) {
    int tok = __ldcg(P.last_token + s);
    if (tok < 0 || tok >= P.V) {
      if (threadIdx.x == 0) raise_flag(P.err, kDevToken);
      tok = 0;
    }
    src = P.embed + static_cast<size_t>(tok) * P.H;
    if (threadIdx.x == 0 && __ldcg(P.len + s) + P.B > P.cap) raise_flag(P.err, kDevCapacity);
  }
  uint4 xs[kMaxIter], gs[kMaxIter];
#pragma unroll
  for (int it = 0; it < kMaxIter; ++it) {
    const int f0 = (it * blockDim.x + threadIdx.x) * 8;
    if (f0 < P.H) {
      xs[it] = *reinterpret_cast<const uint4*>(src + f0);
      gs[it] = *reinterpret_cast<const uint4*>(P.gain + f0);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < kMaxIter; ++it) {
    const int f0 = (it * blockDim.x + threadIdx.x) * 8;
    if (f0 >= P.H) continue;
    const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(&xs[it]);
    const __nv_bfloat16* gv = reinterpret_cast<const __nv_bfloat16*>(&gs[it]);
    float x[8];
    __nv_bfloat16 xg[8], xl[8];  // x * gain as a high bf16 and the bf16 of its remainder
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[k] = __bfloat162float(xv[k]);
      const float y = x[k] * __bfloat162float(gv[k]);
      xg[k] = __float2bfloat16_rn(y);
      xl[k] = __float2bfloat16_rn(y - __bfloat162float(xg[k]));
      ss += x[k] * x[k];
    }
    const size_t off = static_cast<size_t>(row) * P.H + f0;
    *reinterpret_cast<float4*>(P.x + off) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(P.x + off + 4) = make_float4(x[4], x[5], x[6], x[7]);
    *reinterpret_cast<uint4*>(P.xg + off) = *reinterpret_cast<const uint4*>(xg);
    *reinterpret_cast<uint4*>(P.xg + off + static_cast<size_t>(P.xg_lo) * P.H) = *reinterpret_cast<const uint4*>(xl);
    if (P.trace) {
      *reinterpret_cast<float4*>(P.trace + off) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(P.trace + off + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  if (threadIdx.x == 0) tl_stamp(tl, kTlExit);
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    P.ss[row] = t;
  }
}

int launch_embed(const EmbedParams& p, int batch, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * p.B);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, embed_kernel, p));
}

// ---------------------------------------------------------------- greedy verification
// Row argmax of the target logits (lowest index on ties), then the longest prefix of
// drafts matching it plus the bonus token (bpdata.com DFlash article, introduction: the
// target accepts the longest valid prefix). Grid (chunks, B, batch): each CTA reduces one
// chunk of one row; the last CTA of a sequence (arrival counter, no waiting) merges the
// chunks and decides the acceptance.
DEV void better(float& bv, int& bi, float ov, int oi) {
  if (ov > bv || (ov == bv && oi < bi)) {
    bv = ov;
    bi = oi;
  }
}

__global__ void __launch_bounds__(256) verify_kernel(const VerifyParams P) {
  unsigned long long* tl = P.tl ? P.tl + static_cast<size_t>((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_VERIFY) << 32) | static_cast<unsigned>(P.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }
  const int chunk = blockIdx.x, i = blockIdx.y, s = blockIdx.z;
  const int B = P.B, V = P.V;
  const float* row = P.logits + (static_cast<size_t>(s) * B + i) * V;
  const int c0 = chunk * P.chunk_len;
  const int c1 = min(V, c0 + P.chunk_len);
  // The chunk into L2 while the kernel before this one finishes. Only a hint: the logits are
  // read after the wait below, and L2 holds whatever that kernel writes meanwhile. (Rows
  // start 16-byte aligned when V is a multiple of 4; chunks are multiples of 1024 logits.)
  if (threadIdx.x == 0 && (V & 3) == 0 && c1 > c0) bulk_prefetch_l2(row + c0, static_cast<uint32_t>(c1 - c0) * 4u);
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) tl_stamp(tl, 5);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  if ((V & 3) == 0) {
    constexpr int U = 8;  // float4 loads in flight per thread before any compare
    const int stride = 4 * blockDim.x;
    for (int base = c0 + 4 * static_cast<int>(threadIdx.x); base < c1; base += U * stride) {
      float4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = base + u * stride;
        q[u] = k < c1 ? __ldcs(reinterpret_cast<const float4*>(row + k))
                      : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int k = base + u * stride;
        better(bv, bi, q[u].x, k);
        better(bv, bi, q[u].y, k + 1);
        better(bv, bi, q[u].z, k + 2);
        better(bv, bi, q[u].w, k + 3);
      }
    }
  } else {
    for (int k = c0 + static_cast<int>(threadIdx.x); k < c1; k += blockDim.x) better(bv, bi, __ldcs(row + k), k);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_down_sync(0xffffffffu, bv, o);
    const int oi = __shfl_down_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  if (threadIdx.x == 0) tl_stamp(tl, kTlExit);
  __shared__ float wv[8];
  __shared__ int wi[8];
  __shared__ int s_last;
  __shared__ int g[16];
  if ((threadIdx.x & 31) == 0) {
    wv[threadIdx.x >> 5] = bv;
    wi[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) better(bv, bi, wv[w], wi[w]);
    const int slot = (s * B + i) * P.chunks + chunk;
    P.part_v[slot] = bv;
    P.part_i[slot] = bi;
    __threadfence();
    const int old = atomicAdd(P.seq_cnt + s, 1);
    s_last = (old == B * P.chunks - 1);
    if (s_last) P.seq_cnt[s] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  {  // row argmax over the chunks: 16 lanes per row, all loads in flight, then a lane tree
    const int r = threadIdx.x >> 4, l16 = threadIdx.x & 15;
    float v = -INFINITY;
    int idx = 0x7fffffff;
    if (r < B) {
      for (int c = l16; c < P.chunks; c += 16) {
        const int slot = (s * B + r) * P.chunks + c;
        better(v, idx, __ldcg(P.part_v + slot), __ldcg(P.part_i + slot));
      }
    }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {   // every lane of the warp takes part
      const float ov = __shfl_down_sync(0xffffffffu, v, o, 16);
      const int oi = __shfl_down_sync(0xffffffffu, idx, o, 16);
      better(v, idx, ov, oi);
    }
    if (r < B && l16 == 0) g[r] = idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = 0;
    while (j < B - 1 && __ldcg(P.drafted + s * (B - 1) + j) == g[j]) ++j;
    const int tau = j + 1;
    P.accept_len[s] = tau;
    P.last_token[s] = g[j];
    for (int k = 0; k < B; ++k) P.committed[s * B + k] = k < tau ? g[k] : -1;
  }
}

int launch_verify(const VerifyParams& p, int batch, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.chunks, p.B, batch);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, verify_kernel, p));
}

// ---------------------------------------------------------------- sampling-mode verification
// Verification when the target samples at temperature T (7minutos.es, "Casos de uso con
// ejemplos", measures the method under sampling). The pages give no accept rule; this is
// standard speculative sampling with the drafter's argmax as a point proposal: accept
// d_{i+1} while u_i < p_i(d_{i+1}), p_i = softmax(z_i / T); at the first rejection (row j)
// sample by inverse CDF with w from p_j without d_{j+1}; with every draft accepted sample
// the bonus token from p_{B-1}. The uniforms are inputs.
//
// Grid (chunks, B, batch): each CTA reduces one chunk of one row to (max, sum of exp) of
// z / T; the last CTA of a sequence merges the chunks of every row, takes the accept
// decisions, finds the chunk in which the cumulative mass of the stop row crosses
// w * (its mass), and scans that chunk with a block-wide prefix sum.
DEV void lse_merge(float& m, float& s, float om, float os) {
  const float M = fmaxf(m, om);
  if (M == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * __expf(m - M)) + (om == -INFINITY ? 0.f : os * __expf(om - M));
  m = M;
}

__global__ void __launch_bounds__(256) verify_sampling_kernel(const VerifySampleParams P) {
  pdl_wait();
  pdl_launch_dependents();
  const int chunk = blockIdx.x, i = blockIdx.y, sq = blockIdx.z;
  const int B = P.B, V = P.V, tid = threadIdx.x;
  const float* row = P.logits + (static_cast<size_t>(sq) * B + i) * V;
  const int c0 = chunk * P.chunk_len, c1 = min(V, c0 + P.chunk_len);
  float m = -INFINITY, sum = 0.f;  // online max and sum of exp(z / T - max) over the chunk
  for (int k = c0 + tid; k < c1; k += blockDim.x) {
    const float t = __ldcg(row + k) * P.inv_temp;
    if (t > m) {
      sum = (m == -INFINITY ? 0.f : sum * __expf(m - t)) + 1.f;
      m = t;
    } else {
      sum += __expf(t - m);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float om = __shfl_down_sync(0xffffffffu, m, o), os = __shfl_down_sync(0xffffffffu, sum, o);
    lse_merge(m, sum, om, os);
  }
  __shared__ float wm[8], ws[8];
  __shared__ int s_last;
  if ((tid & 31) == 0) {
    wm[tid >> 5] = m;
    ws[tid >> 5] = sum;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) lse_merge(m, sum, wm[w], ws[w]);
    const int slot = (sq * B + i) * P.chunks + chunk;
    P.part_m[slot] = m;
    P.part_s[slot] = sum;
    __threadfence();
    const int old = atomicAdd(P.seq_cnt + sq, 1);
    s_last = (old == B * P.chunks - 1);
    if (s_last) P.seq_cnt[sq] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---- last CTA of the sequence: every row's (max, sum), the accept decisions
  __shared__ float rm[16], rs[16], pd[16];
  __shared__ int s_j, s_tok, s_chunk, s_excl;
  __shared__ float s_w, s_mj;
  __shared__ float scan[256];
  {
    const int r = tid >> 4, l16 = tid & 15;
    float mm = -INFINITY, ss = 0.f;
    if (r < B)
      for (int c = l16; c < P.chunks; c += 16) {
        const int slot = (sq * B + r) * P.chunks + c;
        lse_merge(mm, ss, __ldcg(P.part_m + slot), __ldcg(P.part_s + slot));
      }
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
      const float om = __shfl_down_sync(0xffffffffu, mm, o, 16), os = __shfl_down_sync(0xffffffffu, ss, o, 16);
      lse_merge(mm, ss, om, os);
    }
    if (r < B && l16 == 0) {
      rm[r] = mm;
      rs[r] = ss;
      float p = 0.f;
      if (r < B - 1) {
        const int d = __ldcg(P.drafted + sq * (B - 1) + r);
        if (d >= 0 && d < V) {
          p = __expf(__ldcg(P.logits + (static_cast<size_t>(sq) * B + r) * V + d) * P.inv_temp - mm) / ss;
        } else {
          raise_flag(P.err, kDevToken);
        }
      }
      pd[r] = p;
    }
  }
  __syncthreads();
  if (tid == 0) {
    const float* u = P.uniforms + static_cast<size_t>(sq) * B;
    int j = 0;
    while (j < B - 1 && __ldcg(u + j) < pd[j]) ++j;
    const float* zj = P.logits + (static_cast<size_t>(sq) * B + j) * V;
    const int excl = j < B - 1 ? __ldcg(P.drafted + sq * (B - 1) + j) : -1;
    const float mj = rm[j];
    const float e_ex = (excl >= 0 && excl < V) ? __expf(__ldcg(zj + excl) * P.inv_temp - mj) : 0.f;
    float W = __ldcg(u + B - 1) * (rs[j] - e_ex);
    // the chunk in which the cumulative mass of row j (without the rejected draft) passes W
    float acc = 0.f;
    int cs = P.chunks - 1;
    float w_in = INFINITY;  // not crossed (rounding): the last index of the last chunk
    for (int c = 0; c < P.chunks; ++c) {
      const int slot = (sq * B + j) * P.chunks + c;
      const float pm = __ldcg(P.part_m + slot);
      float mc = pm == -INFINITY ? 0.f : __ldcg(P.part_s + slot) * __expf(pm - mj);
      if (excl >= c * P.chunk_len && excl < (c + 1) * P.chunk_len) mc -= e_ex;
      if (W < acc + mc) {
        cs = c;
        w_in = W - acc;
        break;
      }
      acc += mc;
    }
    s_j = j;
    s_excl = excl;
    s_mj = mj;
    s_chunk = cs;
    s_w = w_in;
    s_tok = -1;
  }
  __syncthreads();
  // ---- block-wide scan of the chosen chunk of row j: each thread a contiguous segment
  {
    const int j = s_j, excl = s_excl, cs = max(s_chunk, 0);
    const float mj = s_mj;
    const float* zj = P.logits + (static_cast<size_t>(sq) * B + j) * V;
    const int a0 = cs * P.chunk_len, a1 = min(V, a0 + P.chunk_len);
    const int seg = (a1 - a0 + blockDim.x - 1) / blockDim.x;
    const int b0 = min(a1, a0 + tid * seg), b1 = min(a1, b0 + seg);
    float local = 0.f;
    for (int v = b0; v < b1; ++v)
      if (v != excl) local += __expf(__ldcg(zj + v) * P.inv_temp - mj);
    scan[tid] = local;
    __syncthreads();
    for (int o = 1; o < static_cast<int>(blockDim.x); o <<= 1) {  // inclusive prefix sums
      const float add = tid >= o ? scan[tid - o] : 0.f;
      __syncthreads();
      scan[tid] += add;
      __syncthreads();
    }
    const float before = scan[tid] - local, Wc = s_w;
    if (Wc >= before && Wc < scan[tid]) {
      float a = before;
      int hit = -1, lastv = -1;
      for (int v = b0; v < b1; ++v) {
        if (v == excl) continue;
        lastv = v;
        a += __expf(__ldcg(zj + v) * P.inv_temp - mj);
        if (Wc < a) {
          hit = v;
          break;
        }
      }
      s_tok = hit >= 0 ? hit : lastv;  // rounding within the segment: its last index
    }
    __syncthreads();
    if (tid == 0 && s_tok < 0) {  // rounding: the last index of the chunk that carries mass
      for (int v = a1 - 1; v >= a0; --v)
        if (v != excl) {
          s_tok = v;
          break;
        }
    }
    __syncthreads();
  }
  if (tid == 0) {
    const int j = s_j, tok = s_tok;
    P.accept_len[sq] = j + 1;
    P.last_token[sq] = tok;
    for (int k = 0; k < B; ++k)
      P.committed[sq * B + k] = k < j ? __ldcg(P.drafted + sq * (B - 1) + k) : (k == j ? tok : -1);
  }
}

int launch_verify_sampling(const VerifySampleParams& p, int batch, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.chunks, p.B, batch);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, verify_sampling_kernel, p));
}

// ---------------------------------------------------------------- fused target-side verification
// The target's final RMSNorm folded into its LM head, as for the drafter's: the operand is
// h * g as two bf16 planes (high, and the bf16 of the remainder) and the LM-head epilogue
// scales each row by 1 / rms(h) from the sum of squares written here. All loads of a
// thread are issued before its stores.
__global__ void __launch_bounds__(256) target_prep_kernel(const TargetPrepParams P) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int kMaxIter = 4;  // Ht <= 4 * 8 * blockDim
  const int row = blockIdx.x;
  const __nv_bfloat16* src = P.hidden + static_cast<size_t>(row) * P.Ht;
  uint4 xs[kMaxIter], gs[kMaxIter];
#pragma unroll
  for (int it = 0; it < kMaxIter; ++it) {
    const int f0 = (it * blockDim.x + threadIdx.x) * 8;
    if (f0 < P.Ht) {
      xs[it] = *reinterpret_cast<const uint4*>(src + f0);
      gs[it] = *reinterpret_cast<const uint4*>(P.gain + f0);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < kMaxIter; ++it) {
    const int f0 = (it * blockDim.x + threadIdx.x) * 8;
    if (f0 >= P.Ht) continue;
    const __nv_bfloat16* xv = reinterpret_cast<const __nv_bfloat16*>(&xs[it]);
    const __nv_bfloat16* gv = reinterpret_cast<const __nv_bfloat16*>(&gs[it]);
    __nv_bfloat16 hi[8], lo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float x = __bfloat162float(xv[k]);
      const float y = x * __bfloat162float(gv[k]);
      hi[k] = __float2bfloat16_rn(y);
      lo[k] = __float2bfloat16_rn(y - __bfloat162float(hi[k]));
      ss += x * x;
    }
    const size_t off = static_cast<size_t>(row) * P.Ht + f0;
    *reinterpret_cast<uint4*>(P.xg + off) = *reinterpret_cast<const uint4*>(hi);
    *reinterpret_cast<uint4*>(P.xg + off + static_cast<size_t>(P.xg_lo) * P.Ht) = *reinterpret_cast<const uint4*>(lo);
  }
  __shared__ float red[8];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_down_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    P.ss[row] = t;
  }
}

int launch_target_prep(const TargetPrepParams& p, int rows, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, target_prep_kernel, p));
}

// The longest prefix of drafts equal to the target's greedy tokens, plus the bonus token
// (bpdata.com, introduction): one thread per sequence.
__global__ void accept_kernel(const AcceptParams P) {
  pdl_wait();
  pdl_launch_dependents();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= P.batch) return;
  const int B = P.B;
  const int* g = P.g + static_cast<size_t>(s) * B;
  int j = 0;
  while (j < B - 1 && __ldcg(P.drafted + s * (B - 1) + j) == __ldcg(g + j)) ++j;
  const int tau = j + 1;
  P.accept_len[s] = tau;
  P.last_token[s] = __ldcg(g + j);
  for (int k = 0; k < B; ++k) P.committed[s * B + k] = k < tau ? __ldcg(g + k) : -1;
}

int launch_accept(const AcceptParams& p, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.batch + 127) / 128);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, accept_kernel, p));
}

// ---------------------------------------------------------------- synthetic target (harness)
__global__ void plant_kernel(float* logits, const int* drafted, const uint8_t* masks, int n_steps,
                             const int* step, int batch, int B, int V, float bump, int* saved) {
  pdl_wait();  // the drafts are final once the previous kernel has completed
  pdl_launch_dependents();
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= batch * B) return;
  const int s = k / B, i = k - s * B;
  int st = *step;
  st = ((st % n_steps) + n_steps) % n_steps;
  saved[2 * k] = -1;
  if (i >= B - 1 || !masks[(static_cast<size_t>(st) * batch + s) * B + i]) return;
  const int tok = drafted[s * (B - 1) + i];
  if (tok < 0 || tok >= V) return;
  const size_t off = (static_cast<size_t>(s) * B + i) * V + tok;
  saved[2 * k] = static_cast<int>(off);
  saved[2 * k + 1] = __float_as_int(logits[off]);
  logits[off] += bump;
}

__global__ void unplant_kernel(float* logits, int* step, int n_steps, int batch, int B, const int* saved) {
  pdl_wait();  // the verification reading these logits has completed
  pdl_launch_dependents();
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k < batch * B && saved[2 * k] >= 0) logits[saved[2 * k]] = __int_as_float(saved[2 * k + 1]);
  if (k == 0) *step = (*step + 1) % n_steps;
}

// Both harness kernels are launched with programmatic dependent launch: they can be
// resident before the previous kernel ends and wait for it in pdl_wait().
static cudaLaunchConfig_t small_cfg(int n, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + 255) / 256);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int launch_plant(float* logits, const int* drafted, const uint8_t* masks, int n_steps, const int* step, int batch,
                 int B, int V, float bump, int* saved, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = small_cfg(batch * B, stream, attr);
  return static_cast<int>(
      cudaLaunchKernelEx(&cfg, plant_kernel, logits, drafted, masks, n_steps, step, batch, B, V, bump, saved));
}

int launch_unplant(float* logits, int* step, int n_steps, int batch, int B, const int* saved, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = small_cfg(batch * B, stream, attr);
  return static_cast<int>(cudaLaunchKernelEx(&cfg, unplant_kernel, logits, step, n_steps, batch, B, saved));
}

}  // namespace dfl
