// Flash-attention building blocks of the block-attention kernel (sm_103a).
//
// One warp owns 16 query rows (the block's slots for one query head) and walks key tiles
// (64 or 32 keys) staged in shared memory by TMA: K and V as fp16, each in boxes of NK keys x
// 64 dims (128-byte rows, 128-byte swizzle). S = Q Kᵀ and O += P V run on the tensor cores as
// mma.sync m16n8k16 with fp16 operands and fp32 accumulation, with an online softmax in
// registers in log2 units. fp16 carries 11 significant bits, the same as TF32: the scores
// are the step's most rounding-sensitive quantity (the attention output is a weighted mean
// of values with much cancellation, so small score errors grow in relative terms), and
// fp16 q, K, P and V keep them, and the products with V, at that precision while K and V
// cost 2 bytes per element.
#pragma once

#include "ptx.cuh"

namespace dfl {

constexpr int kAttnKeys = 64;  // keys per tile of the standalone kernel

DEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
DEV void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
DEV void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
DEV uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte address of element (key, d) in an fp16 K or V tile of NK keys: D/64 TMA boxes of NK
// keys x 128 bytes, each written with the 128-byte swizzle (16-byte chunk c of row r lands at
// chunk c ^ (r & 7)).
template <int NK>
DEV uint32_t kv_addr(uint32_t base, int key, int d) {
  const int box = d >> 6, dd = d & 63;
  return base + box * (NK * 128) + key * 128 + ((((dd >> 3) ^ (key & 7))) << 4);
}

template <int D>
struct FaState {
  uint32_t qa[D / 16][4];  // Q fragments (fp16 A operand, one per 16 dims)
  float m[2], l[2];        // running max (log2 units) and sum for rows r0 and r0 + 8
  float o[D / 8][4];       // unnormalised output accumulators
};

// Q rows for one query head: row i (< B) is query[row0 + i][head*D .. +D); rows >= B are zero.
template <int D>
DEV void fa_begin(FaState<D>& st, const __half* q, size_t row0, size_t ld, int head, int B, int lane) {
  const int r0 = lane >> 2, kc = (lane & 3) * 2;
  const __half* q0 = q + (row0 + r0) * ld + static_cast<size_t>(head) * D;
  const __half* q1 = q0 + 8 * ld;
  const bool v0 = r0 < B, v1 = r0 + 8 < B;
  auto ld2 = [](const __half* p) { return __ldcg(reinterpret_cast<const unsigned int*>(p)); };
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int c = kk * 16 + kc;
    st.qa[kk][0] = v0 ? ld2(q0 + c) : 0u;
    st.qa[kk][1] = v1 ? ld2(q1 + c) : 0u;
    st.qa[kk][2] = v0 ? ld2(q0 + c + 8) : 0u;
    st.qa[kk][3] = v1 ? ld2(q1 + c + 8) : 0u;
  }
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
}

// One tile of NK keys (64 or 32) starting at key0 (keys >= nkeys are masked out); kb / vb
// are the shared-memory addresses of the staged fp16 K and V tiles.
template <int D, int NK = kAttnKeys>
DEV void fa_tile(FaState<D>& st, uint32_t kb, uint32_t vb, int key0, int nkeys, float scale_log2, int lane) {
  constexpr int NT_D = D / 8;
  constexpr int NJ = NK / 8;  // 8-key column tiles of the scores
  const int kq = (lane & 3) * 2;
  float sc[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
  // S = Q Kᵀ. ldmatrix hands lane t row t/4, halves 2(t%4)..+1 of each 8 x 8 matrix: with
  // rows = keys and columns = 8 dims that is the B fragment (k = dims, n = keys). Matrices
  // 0..3: keys 0-7 dims lo, keys 0-7 dims hi, keys 8-15 dims lo, keys 8-15 dims hi.
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int np = 0; np < NK / 16; ++np) {
      const int mi = lane >> 3;
      const int key = np * 16 + (mi >> 1) * 8 + (lane & 7);
      const int d = kk * 16 + (mi & 1) * 8;
      uint32_t b[4];
      ldsm_x4(kv_addr<NK>(kb, key, d), b);
      mma_f16_16816(sc[2 * np], st.qa[kk], b[0], b[1]);
      mma_f16_16816(sc[2 * np + 1], st.qa[kk], b[2], b[3]);
    }
  }
  // scale to log2 units, mask keys past the end, online softmax
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int key = key0 + j * 8 + kq + (c & 1);
      const float v = key < nkeys ? sc[j][c] * scale_log2 : -INFINITY;
      sc[j][c] = v;
      mx[c >> 1] = fmaxf(mx[c >> 1], v);
    }
  }
  float corr[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float mnew = fmaxf(st.m[r], mx[r]);
    const float base = mnew == -INFINITY ? 0.f : mnew;
    corr[r] = exp2f(st.m[r] - base);
    st.m[r] = mnew;
    mx[r] = base;
  }
  float ls[2] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float p = exp2f(sc[j][c] - mx[c >> 1]);
      sc[j][c] = p;
      ls[c >> 1] += p;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) st.l[r] = st.l[r] * corr[r] + ls[r];
#pragma unroll
  for (int nt = 0; nt < NT_D; ++nt) {
    st.o[nt][0] *= corr[0];
    st.o[nt][1] *= corr[0];
    st.o[nt][2] *= corr[1];
    st.o[nt][3] *= corr[1];
  }
  // O += P V
#pragma unroll
  for (int kk = 0; kk < NK / 16; ++kk) {
    uint32_t pa[4];
    pa[0] = pack_f16(sc[2 * kk][0], sc[2 * kk][1]);
    pa[1] = pack_f16(sc[2 * kk][2], sc[2 * kk][3]);
    pa[2] = pack_f16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
    pa[3] = pack_f16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
    for (int dp = 0; dp < D / 16; ++dp) {
      const int mi = lane >> 3;
      const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
      const int d = dp * 16 + (mi >> 1) * 8;
      uint32_t b[4];
      ldsm_x4_trans(kv_addr<NK>(vb, key, d), b);
      mma_f16_16816(st.o[2 * dp], pa, b[0], b[1]);
      mma_f16_16816(st.o[2 * dp + 1], pa, b[2], b[3]);
    }
  }
}

// Row sums across the quad of lanes that share a row.
template <int D>
DEV void fa_end(FaState<D>& st) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
  }
}

}  // namespace dfl
