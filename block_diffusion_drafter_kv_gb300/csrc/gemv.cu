// Weight-streaming GEMM for the DFlash draft path on sm_103a (tcgen05 + TMA + TMEM).
//
// At batch 1 every projection of the drafter (context fusion, K/V injection, Q/K/V, O,
// SwiGLU gate/up/down, LM head) multiplies a large bf16 weight by at most 16 activation
// rows: the cost is reading the weight once from HBM. The weight tile (128 output rows x
// 64 k, 16 KB) is the M=128 A operand of tcgen05.mma and the activation rows are the
// N = 16*NB operand, so a single MMA instruction consumes 4 KB of weights. The
// per-projection work that follows (RMSNorm scaling, RoPE, KV-cache append, residual add,
// SiLU gating, LM-head argmax) runs in the epilogue on the fp32 accumulators read back
// from TMEM, so no projection output makes a second trip through HBM.
//
// CTA layout (192 threads, one CTA per SM):
//   warp 0     TMA producer: weight tiles and activation tiles into an S-stage smem ring
//   warp 1     TMEM allocation; lane 0 issues the MMAs (two TMEM accumulators)
//   warps 2-5  epilogue: warp w reads TMEM lanes 32*(w%4)..+31, i.e. tile rows
//
// Work split: units (tile, k-block) are divided evenly over the grid ("stream-K"); a tile
// covered by several CTAs is reduced by the last one to finish it, summing the partials
// in CTA order, so the result is deterministic and the same for any row count.
// With programmatic dependent launch the producer streams the first S weight tiles
// before waiting for the previous kernel, hiding the kernel boundary behind HBM reads.
#include "internal.h"
#include "ptx.cuh"

namespace dfl {

// NB: activation row groups of 16 (ROWS = 16*NB rows per pass). KSUB: 64-wide k-boxes per
// pipeline stage (a stage holds 128 weight rows x 64*KSUB k, so each weight row contributes
// 128*KSUB contiguous bytes per stage). STAGES: depth of the shared-memory ring.
// MINB: CTAs per SM the launch bounds are sized for.
//
// Activations are carried as two bf16 planes, x = hi + lo with hi = bf16(x) and
// lo = bf16(x - hi), so that a bf16 tensor-core product sees x to about 16 significant
// bits: the B tile of a k-box holds the ROWS high rows followed by the ROWS low rows. Up to
// 128 rows one MMA of N = 2*ROWS multiplies both and the epilogue adds the two halves of
// the fp32 accumulator; at 256 rows (N would exceed 256) one MMA per plane accumulates into
// the same columns. The weight bytes streamed are unchanged; the MMA work doubles, which
// costs nothing while the kernel waits on HBM. Operands that are exact in bf16 (the
// target's hidden states) are loaded as the high plane only, with an MMA of N = ROWS.
template <int NB, int KSUB, int STAGES_, int MINB_>
struct GemvCfg {
  static constexpr int ROWS = 16 * NB;                // activation rows of a pass
  static constexpr bool PLANES_IN_N = 2 * ROWS <= 256;  // both planes in one MMA's N
  static constexpr int NCOL = PLANES_IN_N ? 2 * ROWS : ROWS;  // accumulator columns
  static constexpr int KS = KSUB;
  static constexpr int STAGES = STAGES_;
  static constexpr int MINB = MINB_;
  static constexpr int A_SUB = 128 * 64 * 2;          // one 128 x 64 weight sub-tile (16 KB)
  static constexpr int B_PLANE = ROWS * 64 * 2;       // one plane of a ROWS x 64 activation sub-tile
  static constexpr int B_SUB = 2 * B_PLANE;           // both planes
  static constexpr int A_BYTES = KSUB * A_SUB;
  static constexpr int B_BYTES = KSUB * B_SUB;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * NCOL;          // two accumulators (power of two >= 64)
  static constexpr int XLD = 132;                     // padded row of the exchange buffer
  static constexpr int EPI_BYTES = 16 * XLD * 4 + 5 * ROWS * 4;  // xch, inv, best v/i, row pos/seq
  static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 32;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static constexpr uint32_t IDESC2 = idesc_bf16_f32(128, NCOL);  // both planes (PLANES_IN_N)
  static constexpr uint32_t IDESC1 = idesc_bf16_f32(128, ROWS);  // high plane only
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(TMEM_COLS <= 512, "TMEM columns");
  // CTAs of one persistent launch that can share an SM must fit in its TMEM together, or one
  // would wait in tcgen05.alloc for columns held by a CTA that waits for it at a barrier.
  static_assert((233472 / SMEM) * TMEM_COLS <= 512, "co-resident CTAs exceed TMEM");
};

DEV float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }
DEV __nv_bfloat16 f2bf(float v) { return __float2bfloat16_rn(v); }

// 16 values as fp16 (round to nearest even), 32 bytes at p.
DEV void st16_half(__half* p, const float (&v)[16]) {
  uint4 b[2];
  __half2* h = reinterpret_cast<__half2*>(b);
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
  reinterpret_cast<uint4*>(p)[0] = b[0];
  reinterpret_cast<uint4*>(p)[1] = b[1];
}

// CTA whose unit range contains unit u (units split as floor(c*U/G)).
DEV int cta_of_unit(uint32_t u, uint32_t U, int G) {
  return static_cast<int>(((static_cast<uint64_t>(u) + 1) * G + U - 1) / U) - 1;
}
DEV uint32_t unit_begin(int c, uint32_t U, int G) {
  return static_cast<uint32_t>(static_cast<uint64_t>(c) * U / G);
}
// Partial slot of CTA c for tile t: 2c for its first tile, 2c+1 for its last.
DEV int part_slot(int c, int t, uint32_t U, int G, int KB) {
  return (static_cast<int>(unit_begin(c, U, G) / KB) == t) ? 2 * c : 2 * c + 1;
}

DEV int map_of_tile(const GemvParams& P, int t) {
  int i = 0;
  while (i + 1 < P.n_amaps && t >= P.tile_start[i + 1]) ++i;
  return i;
}

// Weight sub-tiles of k-stage ks (KSUB boxes of 64 k each, two 64-row boxes per sub-tile).
template <int KSUB>
DEV void load_a(const GemvParams& P, int t, int ks, uint8_t* dst, uint64_t* bar, uint64_t pol) {
  int m0, m1, r0, r1;
  if (P.pair_mode) {
    m0 = 0; m1 = 1; r0 = t * 64; r1 = t * 64;
  } else {
    const int mi = map_of_tile(P, t);
    m0 = m1 = mi;
    r0 = (t - P.tile_start[mi]) * 128;
    r1 = r0 + 64;
  }
#pragma unroll
  for (int j = 0; j < KSUB; ++j) {
    const int k = (ks * KSUB + j) * 64;
    tma_load_2d(dst + j * 16384, &P.amap[m0], bar, k, r0, pol);
    tma_load_2d(dst + j * 16384 + 8192, &P.amap[m1], bar, k, r1, pol);
  }
}

// Activation sub-tiles of k-stage ks: per k-box the high plane, then (b_lo != 0) the low
// plane b_lo rows further down the same map.
template <int KSUB, int B_SUB, int B_PLANE>
DEV void load_b(const GemvParams& P, int ks, uint8_t* dst, uint64_t* bar, uint64_t pol) {
#pragma unroll
  for (int j = 0; j < KSUB; ++j) {
    const int kb = ks * KSUB + j;
    if (P.b3d) {
      const int tap = kb / P.b_kb_per_tap;
      const int col = (kb - tap * P.b_kb_per_tap) * 64;
      tma_load_3d(dst + j * B_SUB, &P.bmap, bar, col, P.b_row0, tap, pol);
    } else {
      tma_load_2d(dst + j * B_SUB, &P.bmap, bar, kb * 64, P.b_row0, pol);
      if (P.b_lo) tma_load_2d(dst + j * B_SUB + B_PLANE, &P.bmap, bar, kb * 64, P.b_row0 + P.b_lo, pol);
    }
  }
}

// ---------------------------------------------------------------- epilogue helpers
// The epilogue works on one 16-row chunk of a 128-feature tile in the "row layout": thread
// e holds row r = e / 8 and the 16 consecutive features c0 = (e % 8) * 16 .. c0 + 15, so
// that every global load and store it makes is 16 bytes wide. (The accumulator arrives in
// the column layout of tcgen05.ld, thread m = feature, 16 rows; to_rows transposes it.)
struct RowPos {
  int r, c0;
};
DEV RowPos row_pos(int e) { return {e >> 3, (e & 7) * 16}; }

template <int XLD>
DEV void to_rows(const float (&v)[16], int m, int e, float* xch, float (&o)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) xch[j * XLD + m] = v[j];
  named_bar_sync(1, 128);
  const RowPos rp = row_pos(e);
#pragma unroll
  for (int k = 0; k < 16; k += 4) {
    const float4 q = *reinterpret_cast<const float4*>(xch + rp.r * XLD + rp.c0 + k);
    o[k] = q.x;
    o[k + 1] = q.y;
    o[k + 2] = q.z;
    o[k + 3] = q.w;
  }
  named_bar_sync(1, 128);
}

DEV void ld16(const float* p, float (&o)[16]) {
#pragma unroll
  for (int k = 0; k < 16; k += 4) {
    const float4 q = __ldcg(reinterpret_cast<const float4*>(p + k));
    o[k] = q.x;
    o[k + 1] = q.y;
    o[k + 2] = q.z;
    o[k + 3] = q.w;
  }
}
DEV void st16(float* p, const float (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 16; k += 4) *reinterpret_cast<float4*>(p + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
}
// 16 values as bf16 at p and, when lo_off != 0, the bf16 of the remainders at p + lo_off.
DEV void st16_split(__nv_bfloat16* p, size_t lo_off, const float (&v)[16]) {
  uint4 hi[2], lo[2];
  __nv_bfloat16* hv = reinterpret_cast<__nv_bfloat16*>(hi);
  __nv_bfloat16* lv = reinterpret_cast<__nv_bfloat16*>(lo);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    hv[k] = f2bf(v[k]);
    lv[k] = f2bf(v[k] - bf2f(hv[k]));
  }
  reinterpret_cast<uint4*>(p)[0] = hi[0];
  reinterpret_cast<uint4*>(p)[1] = hi[1];
  if (lo_off) {
    reinterpret_cast<uint4*>(p + lo_off)[0] = lo[0];
    reinterpret_cast<uint4*>(p + lo_off)[1] = lo[1];
  }
}
DEV void ld16_bf16(const __nv_bfloat16* p, float (&o)[16]) {
  uint4 q[2];
  q[0] = reinterpret_cast<const uint4*>(p)[0];
  q[1] = reinterpret_cast<const uint4*>(p)[1];
  const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(q);
#pragma unroll
  for (int k = 0; k < 16; ++k) o[k] = bf2f(b[k]);
}

// Sum of squares of a row's 128 features: each lane sums its 16 in order, then the row's
// 8 lanes combine in a fixed tree; lane (e % 8) == 0 holds the total.
DEV float row_sumsq(const float (&w)[16]) {
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) s += w[k] * w[k];
  s += __shfl_down_sync(0xffffffffu, s, 4, 8);
  s += __shfl_down_sync(0xffffffffu, s, 2, 8);
  s += __shfl_down_sync(0xffffffffu, s, 1, 8);
  return s;
}

// RoPE table entries of a row position for this lane's 16 consecutive pair indices.
DEV void rope_tables_row(int pos, int c0, int d, const float* cosT, const float* sinT, float (&cs)[16],
                         float (&sn)[16]) {
  const int half = d >> 1;
  const int fi0 = (c0 & (d - 1)) & (half - 1);
  ld16(cosT + static_cast<size_t>(pos) * half + fi0, cs);
  ld16(sinT + static_cast<size_t>(pos) * half + fi0, sn);
}

// Rotate-half RoPE on a row: feature c pairs with c ^ (d/2) of the same head, which lives
// in lane (e % 8) ^ (d/32) of the same row group.
DEV void rope_row(float (&val)[16], const float (&cs)[16], const float (&sn)[16], int c0, int d) {
  const int half = d >> 1;
  const bool lo = (c0 & (d - 1)) < half;
  const int lx = half >> 4;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float p = __shfl_xor_sync(0xffffffffu, val[k], lx, 8);
    val[k] = lo ? (val[k] * cs[k] - p * sn[k]) : (val[k] * cs[k] + p * sn[k]);
  }
}

// Epilogue inputs of one 16-row chunk that do not depend on the accumulator, loaded before
// the accumulator (and, on a split tile, the other CTAs' partials) so that their global
// round trips overlap: FC / RESID: a = gains of the lane's 16 features, b = the residual the
// tile updates (RESID); KV / QKV: a, b = RoPE cos / sin at the lane's row position.
struct EpiPre {
  bool have;
  float a[16], b[16];
};

template <int NB, int MINB>
DEV void epilogue_prefetch(const GemvParams& P, int t, int ch, int e, const int* s_pos, EpiPre& pre) {
  pre.have = MINB == 1;  // a halved register budget cannot hold them across the wait
  if (!pre.have) return;
  const RowPos rp = row_pos(e);
  const int lr = ch * 16 + rp.r;
  if (P.op == OP_RESID || P.op == OP_FC) {
    ld16_bf16(P.gain + t * 128 + rp.c0, pre.a);
    if (P.op == OP_RESID) {
      const int gr = P.grow0 + lr;
      if (gr < P.n_valid) {
        ld16(P.y + static_cast<size_t>(gr) * P.y_ld + t * 128 + rp.c0, pre.b);
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) pre.b[k] = 0.f;
      }
    }
  } else if (P.op == OP_KV || P.op == OP_QKV) {
    const int mi = map_of_tile(P, t);
    if (P.op == OP_KV ? !(mi & 1) : mi < 2)
      rope_tables_row(max(s_pos[lr], 0), rp.c0, P.d, P.rope_cos, P.rope_sin, pre.a, pre.b);
  }
}

// Epilogue of rows [chunk*16, chunk*16 + 16) of tile t, v in the row layout.
template <int NB>
DEV void epilogue_rows(const GemvParams& P, int t, int chunk, float (&v)[16], int e, const float* s_inv,
                       float* s_bv, int* s_bi, const int* s_pos, const int* s_seq, const EpiPre& pre) {
  const RowPos rp = row_pos(e);
  const int lr = chunk * 16 + rp.r;    // local row
  const int gr = P.grow0 + lr;          // global row
  const int c0 = rp.c0;
  const size_t lo_off = static_cast<size_t>(P.yb_lo) * P.yb_ld;  // low plane of yb (0: none)
  switch (P.op) {
    case OP_PLAIN: {
      if (gr < P.n_valid) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int n = t * 128 + c0 + k;
          if (n < P.n_out) P.y[static_cast<size_t>(P.out_row0 + lr) * P.y_ld + n] = v[k];
        }
      }
    } break;

    case OP_FC: {
      float g[16], w[16];
      if (pre.have) {
#pragma unroll
        for (int k = 0; k < 16; ++k) g[k] = pre.a[k];
      } else {
        ld16_bf16(P.gain + t * 128 + c0, g);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = v[k] * g[k];
      st16_split(P.yb + static_cast<size_t>(P.out_row0 + lr) * P.yb_ld + t * 128 + c0, lo_off, w);
      const float s = row_sumsq(v);
      if ((e & 7) == 0) P.ss_out[t * P.ss_stride + P.out_row0 + lr] = s;
    } break;

    case OP_KV:
    case OP_QKV: {
      // KV: maps (Wk, Wv) per layer; QKV: 0 = q, 1 = k, 2 = v
      const int mi = map_of_tile(P, t);
      const bool is_q = P.op == OP_QKV && mi == 0;
      const bool is_v = P.op == OP_KV ? (mi & 1) : mi == 2;
      const int layer = P.op == OP_KV ? mi >> 1 : P.layer;
      const int feat0 = (t - P.tile_start[mi]) * 128 + c0;  // head*d + j within the map
      float val[16];
      const float inv = s_inv[lr];
#pragma unroll
      for (int k = 0; k < 16; ++k) val[k] = v[k] * inv;
      if (!is_v) {
        if (pre.have) {
          rope_row(val, pre.a, pre.b, c0, P.d);
        } else {
          float cs[16], sn[16];
          rope_tables_row(max(s_pos[lr], 0), c0, P.d, P.rope_cos, P.rope_sin, cs, sn);
          rope_row(val, cs, sn, c0, P.d);
        }
      }
      if (is_q) {
        if (gr < P.n_valid) st16_half(P.qh + static_cast<size_t>(gr) * P.yb_ld + feat0, val);
      } else if (s_pos[lr] >= 0) {
        const size_t row_elems = static_cast<size_t>(P.nkv) * P.d;
        const size_t off =
            (static_cast<size_t>(layer) * P.layer_rows + s_seq[lr]) * row_elems + feat0;
        st16_half((is_v ? P.vc : P.kc) + off, val);
      }
    } break;

    case OP_RESID: {
      float xo[16], g[16];
      if (pre.have) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          xo[k] = pre.b[k];
          g[k] = pre.a[k];
        }
      } else {
        ld16_bf16(P.gain + t * 128 + c0, g);
        if (gr < P.n_valid) {
          ld16(P.y + static_cast<size_t>(gr) * P.y_ld + t * 128 + c0, xo);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) xo[k] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) xo[k] = gr < P.n_valid ? xo[k] + v[k] : 0.f;
      const float s = row_sumsq(xo);
      if (gr < P.n_valid) {
        const size_t off = static_cast<size_t>(gr) * P.y_ld + t * 128 + c0;
        st16(P.y + off, xo);
        if (P.trace) st16(P.trace + off, xo);
        float w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = xo[k] * g[k];
        st16_split(P.yb + static_cast<size_t>(gr) * P.yb_ld + t * 128 + c0, lo_off, w);
        if ((e & 7) == 0) P.ss_out[t * P.ss_stride + gr] = s;
      }
    } break;

    case OP_SWIGLU: {
      // features 0-63 of the tile are gate rows, 64-127 the matching up rows: lanes 0-3 of a
      // row group hold gate values, lanes 4-7 the up values they pair with
      const float inv = s_inv[lr];
      float a[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float val = v[k] * inv;
        const float up = __shfl_xor_sync(0xffffffffu, val, 4, 8);
        a[k] = val / (1.f + __expf(-val)) * up;
      }
      if (c0 < 64 && gr < P.n_valid) st16_split(P.yb + static_cast<size_t>(gr) * P.yb_ld + t * 64 + c0, lo_off, a);
    } break;

    case OP_LMHEAD: {
      const int vid0 = t * 128 + c0;
      const int B = P.rows_per_seq;
      const float inv = s_inv[lr];
      float z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = v[k] * inv;
      if (P.logits && gr < P.n_valid) {
        const int sq = gr / B, i = gr - sq * B;
        if (i >= 1) {
          float* dst = P.logits + (static_cast<size_t>(sq) * (B - 1) + i - 1) * P.vocab + vid0;
          if (vid0 + 16 <= P.vocab && (P.vocab & 3) == 0) {
            st16(dst, z);
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k)
              if (vid0 + k < P.vocab) dst[k] = z[k];
          }
        }
      }
      // running argmax of the row, lowest index on ties
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (vid0 + k < P.vocab && z[k] > bv) {
          bv = z[k];
          bi = vid0 + k;
        }
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) {
        const float ov = __shfl_down_sync(0xffffffffu, bv, off, 8);
        const int oi = __shfl_down_sync(0xffffffffu, bi, off, 8);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if ((e & 7) == 0 && (bv > s_bv[lr] || (bv == s_bv[lr] && bi < s_bi[lr]))) {
        s_bv[lr] = bv;
        s_bi[lr] = bi;
      }
    } break;
  }
}

DEV int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Release-add at GPU scope: the CTA's writes ordered before it (by a CTA barrier) become
// visible to any thread that reads the new count with ld.acquire.gpu.
DEV void red_release_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Grid-wide phase barrier: every CTA arrives once per phase (a release-add) after its
// epilogue work is done; a waiter sees all of that phase's stores. Bounded: false after
// limit_ns.
DEV bool grid_wait(const int* bar, int target, uint64_t limit_ns) {
  if (ld_acquire_gpu(bar) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);
    if (ld_acquire_gpu(bar) >= target) return true;
    if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// Order this thread's generic-proxy global stores before later async-proxy (TMA) reads.
DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Units of phase P are split over the first Gp = min(G, U) CTAs so that every participating
// CTA has at least one unit (the split-tile bookkeeping counts consecutive participants);
// CTAs c >= Gp have none in this phase but still take part in its barrier.
DEV void phase_units(const GemvParams& P, int c, int G, uint32_t& U, uint32_t& u0, uint32_t& u1, int& Gp) {
  U = static_cast<uint32_t>(P.T) * P.KB;
  Gp = static_cast<uint32_t>(G) < U ? G : static_cast<int>(U);
  if (c < Gp) {
    u0 = unit_begin(c, U, Gp);
    u1 = unit_begin(c + 1, U, Gp);
  } else {
    u0 = u1 = U;
  }
}

// Order in which CTA c visits the tiles of its unit range [u0, u1): ascending, except that in
// passes of several row groups (an epilogue of many 16-row chunks) a last tile shared with
// exactly one other CTA (c + 1, whose first tile it is and whose range runs past it) comes
// second when one whole tile lies between. c finishes that tile, and c + 1's part of it is the
// first work c + 1 does, so c can finish it while the whole tile streams: at the end of the
// phase only that tile's epilogue remains, not two tiles' work. (The whole tile and the moved
// one use different accumulators, so the MMAs never wait for the finishing. With more whole
// tiles, or a one-chunk epilogue, the move measured slower.)
struct TileOrder {
  uint32_t u0, u1;
  int ta, tb;
  bool swap;
  DEV int count() const { return u0 < u1 ? tb - ta + 1 : 0; }
  DEV int tile(int j) const { return !swap ? ta + j : j == 0 ? ta : j == 1 ? tb : ta + j - 1; }
};
template <int NB>
DEV TileOrder tile_order(uint32_t u0, uint32_t u1, uint32_t U, int Gp, int c, uint32_t KB) {
  TileOrder o{u0, u1, 0, -1, false};
  if (u0 >= u1) return o;
  o.ta = static_cast<int>(u0 / KB);
  o.tb = static_cast<int>((u1 - 1) / KB);
  const uint32_t tb_end = static_cast<uint32_t>(o.tb + 1) * KB;
  o.swap = NB > 1 && o.tb - o.ta == 2 && u1 < tb_end && c + 1 < Gp && cta_of_unit(tb_end - 1, U, Gp) == c + 1 &&
           unit_begin(c + 2, U, Gp) > tb_end;
  return o;
}
// The k-th unit of the range in visiting order (ascending within a tile).
DEV uint32_t unit_at(const TileOrder& o, uint32_t KB, uint32_t k) {
  if (!o.swap) return o.u0 + k;
  const uint32_t e0 = static_cast<uint32_t>(o.ta + 1) * KB, b1 = static_cast<uint32_t>(o.tb) * KB;
  const uint32_t n0 = e0 - o.u0, n1 = o.u1 - b1;
  if (k < n0) return o.u0 + k;
  if (k < n0 + n1) return b1 + (k - n0);
  return e0 + (k - n0 - n1);
}

// A chain of projection phases in one persistent launch. Phase p+1 reads what phase p
// wrote, so its activation tiles are loaded only after the phase-p grid barrier, but its
// weight tiles are streamed into every free ring stage before that barrier.
template <class C>
__global__ void __launch_bounds__(192, C::MINB) gemv_kernel(const __grid_constant__ GemvChain CH) {
  constexpr int NB = C::ROWS / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  float* xch = reinterpret_cast<float*>(sB + C::STAGES * C::B_BYTES);
  float* s_inv = xch + 16 * C::XLD;
  float* s_bv = s_inv + C::ROWS;
  int* s_bi = reinterpret_cast<int*>(s_bv + C::ROWS);
  int* s_pos = s_bi + C::ROWS;   // per row of the pass: cache position, or -1 if not written
  int* s_seq = s_pos + C::ROWS;  // per row of the pass: its row in a layer of the cache
  uint64_t* full = reinterpret_cast<uint64_t*>(s_seq + C::ROWS);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mdone = tempty + 2;  // completion of every MMA this CTA issued
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mdone + 1);
  int* s_misc = reinterpret_cast<int*>(s_tmem + 1);  // [0] last arrival, [1..2] wait ok by tile parity, [3] phase ok

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int NP = CH.n_phases;
  const uint64_t WL = CH.wait_ns;
  int* err = CH.ph[0].err;
  unsigned long long* tl = CH.tl ? CH.tl + static_cast<size_t>(c) * kTlWords : nullptr;
  if (tl && threadIdx.x == 0) {
    tl[0] = (static_cast<unsigned long long>(TL_GEMV) << 32) | static_cast<unsigned>(CH.tl_id);
    tl[1] = smid();
    tl_stamp(tl, 2);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(mdone, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < NP; ++p) {
      for (int i = 0; i < CH.ph[p].n_amaps; ++i) tma_prefetch_desc(&CH.ph[p].amap[i]);
      tma_prefetch_desc(&CH.ph[p].bmap);
    }
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  if (threadIdx.x == 0) tl_stamp(tl, 3);
  // Every thread but the producer waits for the previous kernel now and then lets the next
  // one start; the producer first streams weights that do not depend on it.
  if (!(warp == 0 && lane == 0)) {
    pdl_wait();
    pdl_launch_dependents();
  }

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t it = 0;  // stages armed with both weight and activation copies, over all phases
      bool ok = true;
      for (int p = 0; p < NP && ok; ++p) {
        const GemvParams& P = CH.ph[p];
        uint32_t U, u0, u1;
        int Gp;
        phase_units(P, c, G, U, u0, u1, Gp);
        const TileOrder ord = tile_order<NB>(u0, u1, U, Gp, c, P.KB);
        const uint32_t n = u1 > u0 ? u1 - u0 : 0;
        const uint32_t pre = n < static_cast<uint32_t>(C::STAGES) ? n : C::STAGES;
        const uint32_t stage_bytes = C::A_BYTES + (P.b_lo ? 2 : 1) * C::KS * C::B_PLANE;
        tl_stamp(tl, 4 + 4 * p);
        if (n == 0 && p > 0) continue;  // nothing to load: run ahead to the next phase's weights
        uint32_t a_only = 0;  // weights do not depend on earlier phases: stream them first
        for (; a_only < pre; ++a_only) {
          const uint32_t i = it + a_only, s = i % C::STAGES, r = i / C::STAGES;
          if (i >= static_cast<uint32_t>(C::STAGES) && !mbar_wait(&empty[s], (r - 1) & 1, WL)) {
            ok = false;
            break;
          }
          const uint32_t u = unit_at(ord, P.KB, a_only);
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          load_a<C::KS>(P, u / P.KB, u % P.KB, sA + s * C::A_BYTES, &full[s], pol_w);
        }
        bool dep_ok = ok;
        if (dep_ok) {
          if (p == 0) {
            pdl_wait();
            pdl_launch_dependents();
          } else {
            dep_ok = grid_wait(CH.bar + p - 1, G + CH.bar_extra, WL);
          }
        }
        tl_stamp(tl, 5 + 4 * p);
        fence_proxy_async_global();
        // activations of the stages armed above (issued even after a failed wait so that
        // every armed stage completes and the drain below cannot stall)
        for (uint32_t k = 0; k < a_only; ++k) {
          const uint32_t u = unit_at(ord, P.KB, k), s = (it + k) % C::STAGES;
          load_b<C::KS, C::B_SUB, C::B_PLANE>(P, u % P.KB, sB + s * C::B_BYTES, &full[s], pol_x);
        }
        it += a_only;
        if (!ok || !dep_ok) {
          ok = false;
          break;
        }
        for (uint32_t k = pre; k < n; ++k) {
          const uint32_t s = it % C::STAGES, r = it / C::STAGES;
          if (!mbar_wait(&empty[s], (r - 1) & 1, WL)) {
            ok = false;
            break;
          }
          const uint32_t u = unit_at(ord, P.KB, k);
          mbar_arrive_expect_tx(&full[s], stage_bytes);
          load_a<C::KS>(P, u / P.KB, u % P.KB, sA + s * C::A_BYTES, &full[s], pol_w);
          load_b<C::KS, C::B_SUB, C::B_PLANE>(P, u % P.KB, sB + s * C::B_BYTES, &full[s], pol_x);
          ++it;
        }
      }
      if (!ok) raise_flag(err, kDevTimeout);
      // drain: every copy this thread issued has landed before the CTA may exit
      const uint32_t first = it > static_cast<uint32_t>(C::STAGES) ? it - C::STAGES : 0;
      for (uint32_t i = first; i < it; ++i)
        if (!mbar_wait(&full[i % C::STAGES], (i / C::STAGES) & 1, WL)) {
          raise_flag(err, kDevTimeout);
          break;
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      uint32_t i = 0;
      int lt = 0;
      bool ok = true;
      for (int p = 0; p < NP && ok; ++p) {
        const GemvParams& P = CH.ph[p];
        uint32_t U, u0, u1;
        int Gp;
        phase_units(P, c, G, U, u0, u1, Gp);
        if (u0 >= u1) continue;
        const TileOrder ord = tile_order<NB>(u0, u1, U, Gp, c, P.KB);
        for (int jt = 0; ok && jt < ord.count(); ++jt, ++lt) {
          const int t = ord.tile(jt);
          const uint32_t ub = max(u0, static_cast<uint32_t>(t) * P.KB);
          const uint32_t ue = min(u1, static_cast<uint32_t>(t + 1) * P.KB);
          const int acc = lt & 1;
          if (lt >= 2 && !mbar_wait(&tempty[acc], ((lt >> 1) - 1) & 1, WL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + acc * C::NCOL;
          const uint32_t idesc = (P.b_lo && C::PLANES_IN_N) ? C::IDESC2 : C::IDESC1;
          const bool lo_mma = P.b_lo && !C::PLANES_IN_N;  // the low plane as a second MMA
          for (uint32_t u = ub; u < ue; ++u, ++i) {
            const uint32_t s = i % C::STAGES, r = i / C::STAGES;
            if (!mbar_wait(&full[s], r & 1, WL)) {
              ok = false;
              break;
            }
            if (u == u0) tl_stamp(tl, 6 + 4 * p);
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * C::A_BYTES);
            const uint32_t b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int j = 0; j < C::KS; ++j)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc_k_sw128(a0 + j * C::A_SUB + kk * 32);
                tc_mma_bf16(d_tmem, ad, smem_desc_k_sw128(b0 + j * C::B_SUB + kk * 32), idesc,
                            (u > ub || j > 0 || kk > 0) ? 1u : 0u);
                if (lo_mma) tc_mma_bf16(d_tmem, ad, smem_desc_k_sw128(b0 + j * C::B_SUB + C::B_PLANE + kk * 32), idesc, 1u);
              }
            tc_commit(&empty[s]);
          }
          if (ok) tc_commit(&tfull[acc]);
        }
      }
      if (!ok) raise_flag(err, kDevTimeout);
      // Every MMA issued has completed before TMEM is released at the end of the kernel.
      // (Normally the epilogue has already waited for them; after an abandoned wait it may
      // not have.)
      tc_commit(mdone);
      if (!mbar_wait(mdone, 0, WL)) raise_flag(err, kDevTimeout);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int e = threadIdx.x - 64;
    const int q = warp & 3;
    const int m = q * 32 + lane;
    int lt = 0;
    bool alive = true;
    for (int p = 0; p < NP && alive; ++p) {
      const GemvParams& P = CH.ph[p];
      uint32_t U, u0, u1;
      int Gp;
      phase_units(P, c, G, U, u0, u1, Gp);
      if (p > 0) {
        if (e == 0) s_misc[3] = grid_wait(CH.bar + p - 1, G + CH.bar_extra, WL) ? 1 : 0;
        named_bar_sync(1, 128);
        if (!s_misc[3]) {
          if (e == 0) raise_flag(err, kDevTimeout);
          alive = false;
          break;
        }
      }
      if (P.ss_in) {
        // inv_rms of every row of the pass: 8 lanes per row each sum a strided subset of the
        // per-tile partials (all loads in flight at once), then a fixed lane tree combines them.
        for (int r0 = 0; r0 < C::ROWS; r0 += 16) {
          const int r = r0 + (e >> 3), lane8 = e & 7;
          const float* src = P.ss_in + P.ss_row0 + r;
          float part = 0.f;
#pragma unroll 4
          for (int pp = lane8; pp < P.ss_parts; pp += 8) part += __ldcg(src + static_cast<size_t>(pp) * P.ss_stride);
          part += __shfl_down_sync(0xffffffffu, part, 4, 8);
          part += __shfl_down_sync(0xffffffffu, part, 2, 8);
          part += __shfl_down_sync(0xffffffffu, part, 1, 8);
          if (lane8 == 0) s_inv[r] = rsqrtf(part / static_cast<float>(P.H) + P.eps);
        }
      }
      for (int r = e; r < C::ROWS; r += 128) {
        s_bv[r] = -INFINITY;
        s_bi[r] = 0x7fffffff;
        if (P.op == OP_KV || P.op == OP_QKV) {  // where each row of the pass goes in the cache
          const int gr = P.grow0 + r;
          const int sq = gr / P.rows_per_seq, i = gr - sq * P.rows_per_seq;
          int pos = -1;
          if (P.op == OP_KV ? (sq < P.batch && i < __ldcg(P.n_new + sq)) : (gr < P.n_valid)) {
            pos = __ldcg(P.len + sq) + i;
            if (pos >= P.cap) {
              raise_flag(P.err, kDevCapacity);
              pos = -1;
            }
          }
          // the row of this position in a layer of the cache: sequence-major, or through the
          // sequence's page table (pages of kPageRows positions)
          int crow = -1;
          if (pos >= 0) {
            if (P.page_table) {
              const int page = __ldcg(P.page_table + static_cast<size_t>(sq) * P.pages_per_seq + pos / kPageRows);
              if (page < 0 || page >= P.layer_rows / kPageRows) {
                raise_flag(P.err, kDevCapacity);
                pos = -1;
              } else {
                crow = page * kPageRows + (pos & (kPageRows - 1));
              }
            } else {
              crow = sq * P.cap + pos;
            }
          }
          s_pos[r] = pos;
          s_seq[r] = crow;
        }
      }
      named_bar_sync(1, 128);
      const bool split = P.b_lo != 0 && C::PLANES_IN_N;  // planes in separate accumulator columns
      // Accumulator of 16 rows (chunk ch): high-plane columns, plus the low-plane columns.
      auto tmem_ld_acc = [&](uint32_t taddr, int ch, bool two, float (&v)[16]) {
        tmem_ld16(taddr + ch * 16, v);
        if (two) {
          float w[16];
          tmem_ld16(taddr + C::ROWS + ch * 16, w);
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] += w[j];
        }
      };
      if (u0 < u1) {
        const TileOrder ord = tile_order<NB>(u0, u1, U, Gp, c, P.KB);
        for (int jt = 0; jt < ord.count(); ++jt, ++lt) {
          const int t = ord.tile(jt);
          const int acc = lt & 1;
          EpiPre pre;
          epilogue_prefetch<NB, C::MINB>(P, t, 0, e, s_pos, pre);
          if (e == 0) s_misc[1 + acc] = mbar_wait(&tfull[acc], (lt >> 1) & 1, WL) ? 1 : 0;
          named_bar_sync(1, 128);
          if (!s_misc[1 + acc]) {
            if (e == 0) raise_flag(err, kDevTimeout);
            alive = false;
            break;
          }
          tc_fence_after();
          const int ca = cta_of_unit(static_cast<uint32_t>(t) * P.KB, U, Gp);
          const int cb = cta_of_unit(static_cast<uint32_t>(t + 1) * P.KB - 1, U, Gp);
          const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * C::NCOL;
          // The CTA whose last tile this is finishes it alone (keeping its own sum in TMEM)
          // with one row group, and with several when one other CTA shares the tile and
          // runs past its end (no CTA lies wholly inside it): then nobody else finishes.
          const bool solo = c == ca && (NB == 1 || (C::MINB == 1 && cb == ca + 1 &&
                                                     unit_begin(cb + 1, U, Gp) > static_cast<uint32_t>(t + 1) * P.KB));
          if (ca == cb) {
            for (int ch = 0; ch < NB; ++ch) {
              float v[16], w[16];
              if (ch > 0) epilogue_prefetch<NB, C::MINB>(P, t, ch, e, s_pos, pre);
              tmem_ld_acc(taddr, ch, split, v);
              if (ch == NB - 1) {
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
              }
              to_rows<C::XLD>(v, m, e, xch, w);
              epilogue_rows<NB>(P, t, ch, w, e, s_inv, s_bv, s_bi, s_pos, s_seq, pre);
            }
          } else if (!solo) {
            // split tile, contributor (with several row groups, every CTA of the tile unless
            // the tile has a sole finisher): its partial goes to its slot ([ROWS][128] fp32,
            // row layout), then it is counted in
            const int slot = part_slot(c, t, U, Gp, P.KB);
            float* dst = P.part + static_cast<size_t>(slot) * C::ROWS * 128;
            const RowPos rp = row_pos(e);
            for (int ch = 0; ch < NB; ++ch) {
              float v[16], w[16];
              tmem_ld_acc(taddr, ch, split, v);
              if (ch == NB - 1) {
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
              }
              to_rows<C::XLD>(v, m, e, xch, w);
              st16(dst + (ch * 16 + rp.r) * 128 + rp.c0, w);
            }
            // the CTA barrier orders every thread's partial before thread 0's release
            named_bar_sync(1, 128);
            if (e == 0) red_release_gpu(P.tile_cnt + t, 1);
            if (NB > 1) {
              // Several row groups: the finishing is shared. Every CTA of the tile whose last
              // tile this is (ca and the CTAs wholly inside it, all done with their units at
              // about the same time) waits for every partial, then finishes row chunks
              // ch = k, k + n_sh, ... (k = c - ca), adding the partials in CTA order.
              const uint32_t tile_end = static_cast<uint32_t>(t + 1) * P.KB;
              if (unit_begin(c + 1, U, Gp) <= tile_end) {
                const int n_c = cb - ca + 1;
                const int n_sh = (unit_begin(cb + 1, U, Gp) <= tile_end ? cb : cb - 1) - ca + 1;
                if (e == 0) {
                  const bool ok = grid_wait(P.tile_cnt + t, n_c, WL);
                  // each sharer counts itself past the partials; the last clears the counter
                  if (ok && atomicAdd(P.tile_cnt + t, 1) == n_c + n_sh - 1) P.tile_cnt[t] = 0;
                  s_misc[0] = ok ? 1 : 0;
                }
                named_bar_sync(1, 128);
                if (!s_misc[0]) {
                  if (e == 0) raise_flag(err, kDevTimeout);
                  alive = false;
                  break;
                }
                constexpr int PR = C::MINB == 1 ? 6 : 4;
                for (int ch = c - ca; ch < NB; ch += n_sh) {
                  EpiPre pc;
                  epilogue_prefetch<NB, C::MINB>(P, t, ch, e, s_pos, pc);
                  auto part_row = [&](int cc) {
                    return P.part + static_cast<size_t>(part_slot(cc, t, U, Gp, P.KB)) * C::ROWS * 128 +
                           (ch * 16 + rp.r) * 128 + rp.c0;
                  };
                  float v[16];
                  ld16(part_row(ca), v);
                  for (int cc0 = ca + 1; cc0 <= cb; cc0 += PR) {
                    float a[PR][16];
#pragma unroll
                    for (int q2 = 0; q2 < PR; ++q2)
                      if (cc0 + q2 <= cb) ld16(part_row(cc0 + q2), a[q2]);
#pragma unroll
                    for (int q2 = 0; q2 < PR; ++q2)
                      if (cc0 + q2 <= cb) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] += a[q2][k];
                      }
                  }
                  epilogue_rows<NB>(P, t, ch, v, e, s_inv, s_bv, s_bi, s_pos, s_seq, pc);
                }
              }
            }
          } else {
            // split tile, sole finisher: CTA ca, whose last tile this is. The others reach it
            // first (cb) or only (CTAs in between), so ca is usually the last to get here; it
            // keeps its own sum, waits for the cb - ca other partials and adds them in CTA
            // order.
            const RowPos rp = row_pos(e);
            float own[16];
            if constexpr (NB == 1) {  // own accumulator out of TMEM while the others finish
              float v[16];
              tmem_ld_acc(taddr, 0, split, v);
              tc_fence_before();
              mbar_arrive(&tempty[acc]);
              to_rows<C::XLD>(v, m, e, xch, own);
            }
            if (e == 0) {
              const bool ok = grid_wait(P.tile_cnt + t, cb - ca, WL);
              if (ok) P.tile_cnt[t] = 0;
              s_misc[0] = ok ? 1 : 0;
            }
            named_bar_sync(1, 128);
            if (!s_misc[0]) {
              if (e == 0) raise_flag(err, kDevTimeout);
              if (NB != 1) {
                tc_fence_before();
                mbar_arrive(&tempty[acc]);
              }
              alive = false;
              break;
            }
            // the poller's ld.acquire.gpu plus the CTA barrier order the partial loads after
            // the contributors' releases
            if constexpr (NB > 1) {
              // one other partial (cb = ca + 1), its rows loaded AH chunks ahead of the chunk
              // being finished so that the chunks' global round trips overlap
              const float* pb = P.part + static_cast<size_t>(part_slot(cb, t, U, Gp, P.KB)) * C::ROWS * 128 +
                                rp.r * 128 + rp.c0;
              constexpr int AH = NB >= 8 ? 2 : 1;  // chunks loaded ahead (registers allowing)
              float a0[16], a1[16];
              ld16(pb, a0);
              if (AH == 2) ld16(pb + 16 * 128, a1);
              for (int ch = 0; ch < NB; ++ch) {
                float a2[16];
                if (ch + AH < NB) {
                  ld16(pb + (ch + AH) * 16 * 128, a2);
                } else {
#pragma unroll
                  for (int k = 0; k < 16; ++k) a2[k] = 0.f;
                }
                if (ch > 0) epilogue_prefetch<NB, C::MINB>(P, t, ch, e, s_pos, pre);
                float a0t[16], v[16];
                tmem_ld_acc(taddr, ch, split, a0t);
                if (ch == NB - 1) {
                  tc_fence_before();
                  mbar_arrive(&tempty[acc]);
                }
                to_rows<C::XLD>(a0t, m, e, xch, v);
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] += a0[k];
                epilogue_rows<NB>(P, t, ch, v, e, s_inv, s_bv, s_bi, s_pos, s_seq, pre);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                  if (AH == 2) {
                    a0[k] = a1[k];
                    a1[k] = a2[k];
                  } else {
                    a0[k] = a2[k];
                  }
                }
              }
            } else {
              // one row group: the others' partials, up to PR CTAs' loads in flight per round
              constexpr int PR = C::MINB == 1 ? 8 : 4;
              auto part_row = [&](int cc) {
                return P.part + static_cast<size_t>(part_slot(cc, t, U, Gp, P.KB)) * C::ROWS * 128 + rp.r * 128 + rp.c0;
              };
              float v[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] = own[k];
              for (int cc0 = ca + 1; cc0 <= cb; cc0 += PR) {
                float a[PR][16];
#pragma unroll
                for (int q2 = 0; q2 < PR; ++q2)
                  if (cc0 + q2 <= cb) ld16(part_row(cc0 + q2), a[q2]);
#pragma unroll
                for (int q2 = 0; q2 < PR; ++q2)
                  if (cc0 + q2 <= cb) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) v[k] += a[q2][k];
                  }
              }
              epilogue_rows<NB>(P, t, 0, v, e, s_inv, s_bv, s_bi, s_pos, s_seq, pre);
            }
          }
        }
      }
      if (!alive) break;

      // ---------------------------------------------- phase-level completion hooks
      if (P.op == OP_LMHEAD || (P.op == OP_KV && P.commit_len)) {
        named_bar_sync(1, 128);
        if (P.op == OP_LMHEAD) {
          for (int r = e; r < C::ROWS; r += 128) {
            P.best_v[c * kMaxPassRows + r] = s_bv[r];
            P.best_i[c * kMaxPassRows + r] = s_bi[r];
          }
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (e == 0) {
          const int old = atomicAdd(P.cta_cnt, 1);
          const int last = (old == G - 1);
          if (last) *P.cta_cnt = 0;
          s_misc[0] = last;
        }
        named_bar_sync(1, 128);
        if (s_misc[0]) {
          __threadfence();
          if (P.op == OP_LMHEAD) {
            const int B = P.rows_per_seq;
            for (int r0 = 0; r0 < C::ROWS; r0 += 16) {
              const int r = r0 + (e >> 3), lane8 = e & 7;
              float bv = -INFINITY;
              int bi = 0x7fffffff;
              // the CTAs' candidates for row r, 160 at a time (one round up to 160 CTAs): all
              // loads of a round in flight at once, then compared in CTA order
              constexpr int kPer = 20;
              for (int c0 = 0; c0 < G; c0 += 8 * kPer) {
                float ov[kPer];
                int oi[kPer];
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                  const int cc = c0 + lane8 + 8 * k;
                  ov[k] = cc < G ? __ldcg(P.best_v + cc * kMaxPassRows + r) : -INFINITY;
                  oi[k] = cc < G ? __ldcg(P.best_i + cc * kMaxPassRows + r) : 0x7fffffff;
                }
#pragma unroll
                for (int k = 0; k < kPer; ++k)
                  if (ov[k] > bv || (ov[k] == bv && oi[k] < bi)) { bv = ov[k]; bi = oi[k]; }
              }
#pragma unroll
              for (int off = 4; off >= 1; off >>= 1) {
                const float ov = __shfl_down_sync(0xffffffffu, bv, off, 8);
                const int oi = __shfl_down_sync(0xffffffffu, bi, off, 8);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
              }
              const int gr = P.grow0 + r;
              if (lane8 == 0 && gr < P.n_valid) {
                const int s = gr / B, i = gr - s * B;
                if (P.lm_all_rows) P.drafted[gr] = bi;
                else if (i >= 1) P.drafted[s * (B - 1) + i - 1] = bi;
              }
            }
          } else {
            for (int s = e; s < P.batch; s += 128) {
              const int nl = __ldcg(P.len + s) + __ldcg(P.n_new + s);
              P.len[s] = nl < P.cap ? nl : P.cap;
            }
          }
        }
      }
      // ---------------------------------------------- arrive at this phase's barrier
      fence_proxy_async_global();
      named_bar_sync(1, 128);
      if (e == 0) {
        tl_stamp(tl, 7 + 4 * p);
        red_release_gpu(CH.bar + p, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (threadIdx.x == 0) {  // the last CTA out clears the barrier counters for the next launch
    tl_stamp(tl, kTlExit);
    __threadfence();
    if (atomicAdd(CH.exit_cnt, 1) == G - 1) {
      for (int p = 0; p < NP; ++p) CH.bar[p] = 0;
      *CH.exit_cnt = 0;
      __threadfence();
    }
  }
}


template <class C>
static int launch_cfg(const GemvChain& p, int n_ctas, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, gemv_kernel<C>, p));
}

template <class C>
static int set_attr() {
  return static_cast<int>(cudaFuncSetAttribute(gemv_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
}

// Kernel variants: row groups NB, k-boxes per stage, ring depth, CTAs per SM.
#define DFL_GEMV_VARIANTS(X)   \
  X(0, 1, 1, 5, 2)              \
  X(1, 1, 1, 10, 1)             \
  X(2, 1, 2, 5, 1)              \
  X(3, 1, 4, 2, 1)              \
  X(4, 1, 2, 4, 1)              \
  X(5, 1, 2, 2, 2)              \
  X(6, 2, 1, 4, 2)              \
  X(7, 4, 1, 3, 2)              \
  X(8, 8, 1, 3, 1)              \
  X(9, 2, 4, 2, 1)              \
  X(10, 4, 2, 3, 1)             \
  X(11, 8, 2, 2, 1)             \
  X(12, 16, 1, 2, 1)

// Several k-boxes per stage for every row count (contiguous bytes per weight row, and about
// 128 KB of weights in flight per SM where shared memory allows); the 1-box variants 0 and
// 6..8 serve phases whose k-block count the box count does not divide.
int gemv_variant(int nb, int pref) {
  if (nb == 1) return (pref >= 0 && pref <= 5) ? pref : 3;
  return nb == 2 ? 9 : nb == 4 ? 10 : nb == 8 ? 11 : 12;
}

int gemv_variant_ksub1(int nb) { return nb == 1 ? 0 : nb == 2 ? 6 : nb == 4 ? 7 : nb == 8 ? 8 : 12; }

int gemv_variant_ksub(int v) {
#define DFL_KS(ID, NB, KS, ST, MB) if (v == ID) return KS;
  DFL_GEMV_VARIANTS(DFL_KS)
#undef DFL_KS
  return 1;
}

int gemv_set_attributes() {
  int e = 0;
#define DFL_SET(ID, NB, KS, ST, MB) if (e == 0) e = set_attr<GemvCfg<NB, KS, ST, MB>>();
  DFL_GEMV_VARIANTS(DFL_SET)
#undef DFL_SET
  return e;
}

int launch_gemv(const GemvChain& p, int variant, int n_ctas, cudaStream_t stream, bool pdl) {
#define DFL_LAUNCH(ID, NB, KS, ST, MB) \
  if (variant == ID) return launch_cfg<GemvCfg<NB, KS, ST, MB>>(p, n_ctas, stream, pdl);
  DFL_GEMV_VARIANTS(DFL_LAUNCH)
#undef DFL_LAUNCH
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace dfl
