// Fused linear cross-entropy: logits = H W^T (+ bias) formed tile by tile on
// the tensor cores and never stored.
//
// Forward (Liger-Kernel issue #533 "Gradient checkpointing for grad_weight in
// LFCE": chunked logits; the fully recomputed variant of its follow-up
// comments keeps no gradient from the forward): one persistent tcgen05 GEMM
// over (token tile, vocab tile) pairs whose epilogue turns each 128 x BN
// logits tile into a per-row partial (max, sum of exp) in the base-2 domain
// and picks out the label logit; a combine kernel merges the partials of a row
// in a fixed order into lse_i and loss_i; the shared finalize kernel reduces.
//
// Backward, per chunk of C rows:
//   1. the same GEMM recomputes the logits of the chunk; its epilogue forms
//      dZ = valid (exp(z - lse) - onehot) g scale and writes it, rounded to the
//      input dtype, to a [C, ldV] workspace buffer (Liger's feature pitch
//      casts the chunk's gradient to the input dtype before the addmm);
//   2. grad_bias += column sums of dZ, in a fixed order without atomics:
//      partial sums per 32 rows, formed by the dZ epilogue from its staged
//      tiles (eight epilogue warps, K <= 1024) or by a pass over the stored
//      dZ, then added up by the epilogue warps of step 3 (or 4) before their
//      first tile;
//   3. grad_H[chunk] = dZ W                (A = dZ K-major, B = W MN-major);
//   4. grad_W (+)= dZ^T H[chunk] in fp32   (A = dZ MN-major, B = H MN-major),
//      the addmm with beta = 1 of the same page, chunk after chunk.
// The tf32 tensor-core path (fp32 inputs) reads K-major operands only, so for
// fp32 the MN-major operands of steps 3 and 4 are first transposed into the
// workspace (W once per call, dZ and H[chunk] once per chunk).  When a chunk
// has too few grad_H tiles to fill the GPU, step 3 splits its long K (= V)
// and the fp32 partials are added in a fixed order (by step 4's epilogue
// warps before their first tile, or by a kernel).  The dZ recompute and grad_W
// run on CTA pairs (tc_gemm_pair_kernel) by default; flce_gemm_set_pair
// selects per contraction.
//
// Also here: the fused forward + backward (flce_fwd_bwd: the forward epilogue
// keeps the chunk's logits as offsets from each tile's maximum, dZ is formed
// from them in place, 6NDV flops in all), the vocabulary-parallel entry points
// (flce_fwd_shard / flce_bwd_shard and the rescale / finish kernels of the
// cross-rank merge) and the raw contraction flce_gemm.
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/flce_gemm.h"
#include "host.h"
#include "tc_gemm.cuh"

namespace flce {

// ----------------------------------------------------------------- epilogues

// v[j] += bias[col0 + j] for the columns inside the vocabulary: 16-byte loads
// when all 32 columns are inside and aligned (the address is the same for the
// whole warp, so each load is one broadcast), element loads otherwise.
template <typename T>
__device__ __forceinline__ void add_bias32(const void* bias, int col0, int V, float (&v)[32]) {
  const T* b = static_cast<const T*>(bias) + col0;
  if (col0 + 32 <= V && (reinterpret_cast<uintptr_t>(b) & 15u) == 0) {
    constexpr int EPV = Elem<T>::kPerVec;
    const uint4* bv = reinterpret_cast<const uint4*>(b);
#pragma unroll
    for (int k = 0; k < 32 / EPV; ++k) {
      float x[EPV];
      Elem<T>::unpack(__ldg(bv + k), x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) v[k * EPV + e] += x[e];
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < V) v[j] += Elem<T>::load(b + j);
  }
}

// The bias of one 32-column chunk, fetched a chunk ahead of its use so that
// the loads are in flight while the previous chunk is reduced (an epilogue
// warp has no other warp on its scheduler to hide their latency).  Only whole,
// aligned chunks are fetched; add_bias32 takes the others element by element.
template <typename T>
struct BiasAhead {
  static constexpr int kVecs = 32 / Elem<T>::kPerVec;
  uint4 w[kVecs];
  __device__ static bool vec_ok(const void* bias, int col0, int V) {
    return col0 + 32 <= V &&
           (reinterpret_cast<uintptr_t>(static_cast<const T*>(bias) + col0) & 15u) == 0;
  }
  __device__ void fetch(const void* bias, int col0, int V) {
    if (vec_ok(bias, col0, V)) {
      const uint4* bv = reinterpret_cast<const uint4*>(static_cast<const T*>(bias) + col0);
#pragma unroll
      for (int k = 0; k < kVecs; ++k) w[k] = __ldg(bv + k);
    }
  }
  __device__ void add(const void* bias, int col0, int V, float (&v)[32]) const {
    if (vec_ok(bias, col0, V)) {
      constexpr int EPV = Elem<T>::kPerVec;
#pragma unroll
      for (int k = 0; k < kVecs; ++k) {
        float x[EPV];
        Elem<T>::unpack(w[k], x);
#pragma unroll
        for (int e = 0; e < EPV; ++e) v[k * EPV + e] += x[e];
      }
    } else {
      add_bias32<T>(bias, col0, V, v);
    }
  }
};

// Adds the first n (<= 32) of 32 logits v to a base-2 online log-sum-exp: the
// chunk maximum (the order of v equals the order of v*log2e), one rescale,
// then 2^(v*log2e - m) by packed pairs (FFMA2) summed into four independent
// packed accumulators, so the sum is not one long chain of dependent adds.
__device__ __forceinline__ void lse_add32(const float (&v)[32], int n, Lse2& st) {
  float mx = -INFINITY;
  if (n >= 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = fmaxf(mx, v[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) mx = fmaxf(mx, v[j]);
  }
  const float bm = mx * kLog2e;
  if (bm > st.m) {
    st.s *= ex2(st.m - bm);
    st.m = bm;
  }
  if (st.m == -INFINITY) return;
  const float2 lg = make_float2(kLog2e, kLog2e), nm = make_float2(-st.m, -st.m);
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), lg, nm);
    float2 e = make_float2(ex2(t.x), ex2(t.y));
    if (n < 32) {
      e.x = j < n ? e.x : 0.0f;
      e.y = j + 1 < n ? e.y : 0.0f;
    }
    acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], e);
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  st.s += a.x + a.y;
}

// As lse_add32, for 32 values already in the base-2 domain (t = z log2(e)).
__device__ __forceinline__ void lse_add32_base2(const float (&t)[32], int n, Lse2& st) {
  float mx = -INFINITY;
  if (n >= 32) {
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = fmaxf(mx, t[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) mx = fmaxf(mx, t[j]);
  }
  if (mx > st.m) {
    st.s *= ex2(st.m - mx);
    st.m = mx;
  }
  if (st.m == -INFINITY) return;
  const float2 nm = make_float2(-st.m, -st.m);
  float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                   make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 u = __fadd2_rn(make_float2(t[j], t[j + 1]), nm);
    float2 e = make_float2(ex2(u.x), ex2(u.y));
    if (n < 32) {
      e.x = j < n ? e.x : 0.0f;
      e.y = j + 1 < n ? e.y : 0.0f;
    }
    acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], e);
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  st.s += a.x + a.y;
}

// The bias of 8 consecutive columns from col0 (those at or past V read as 0):
// one 16-byte load (bf16) or two (fp32) when the 8 lie inside and aligned.
template <typename T>
__device__ __forceinline__ void bias8(const T* bias, int col0, int V, float (&x)[8]) {
  const T* b = bias + col0;
  if (col0 + 8 <= V && (reinterpret_cast<uintptr_t>(b) & 15u) == 0) {
    constexpr int EPV = Elem<T>::kPerVec;
#pragma unroll
    for (int k = 0; k < 8 / EPV; ++k) {
      float y[EPV];
      Elem<T>::unpack(__ldg(reinterpret_cast<const uint4*>(b) + k), y);
#pragma unroll
      for (int e = 0; e < EPV; ++e) x[k * EPV + e] = y[e];
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = col0 + e < V ? Elem<T>::load(b + e) : 0.0f;
  }
}

// v[j] for the one j with base + j == idx (idx in [base, base + 32)).
__device__ __forceinline__ float pick32(const float (&v)[32], int64_t idx, int base) {
  float r = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (base + j == idx) r = v[j];
  return r;
}

// Forward: per-row partial log-sum-exp of one logits tile + label gather.
template <typename T>
struct EpiLse {
  struct Params {
    const void* bias;  // [V] of T or null
    const int64_t* labels;
    int64_t ignore_index;
    int M, V;          // V: columns of this (shard of the) vocabulary
    int64_t part_ld;   // row stride of part_m / part_s (>= M)
    float* part_m;     // [nNt, part_ld], base-2 max
    float* part_s;     // [nNt, part_ld], sum of 2^(t - max)
    float* zlab;       // [M] label logit (written by the tile holding the label)
    int64_t v0;        // vocabulary id of this shard's column 0 (0 unsharded)
    int32_t* status = nullptr;  // device status word (index checks of checked builds)
  };
  template <int BN>
  __device__ static void tile(const Params& p, int mt, int nt, int row_in_tile, uint32_t taddr,
                              EpiCtx& ctx) {
    static_assert(BN == 256, "one bias value per lane and 8-column group");
    const int row = mt * kBM + row_in_tile;
    const bool row_ok = row < p.M;
    const int64_t y = row_ok ? p.labels[row] : -1;
    const int col_base = nt * BN;
    const int64_t ylocal = (y < 0) ? -1 : (y - p.v0) - col_base;
    const T* bias = static_cast<const T*>(p.bias);
    const int lane = row_in_tile & 31;
    // The tile's bias as fp32 times log2(e) in this warp's staging buffer
    // (this epilogue stores nothing through it; two halves, this tile's and
    // the next one's): each logit then costs one FFMA, t = z log2(e) +
    // b log2(e).  The next tile's bias is loaded while this tile is reduced.
    const float* b2 = nullptr;
    float nb[8];
    const bool fetch_next = bias != nullptr && ctx.next_nt >= 0 && ctx.next_nt != nt;
    if (bias != nullptr) {
      float* sb = reinterpret_cast<float*>(ctx.buf);
      if (ctx.aux_nt != nt) {  // not fetched ahead (the CTA's first tile)
        float x[8];
        bias8<T>(bias, col_base + 8 * lane, p.V, x);
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 8; ++e) sb[ctx.aux * BN + 8 * lane + e] = x[e] * kLog2e;
        __syncwarp();
        ctx.aux_nt = nt;
      }
      b2 = sb + ctx.aux * BN;
      if (fetch_next) bias8<T>(bias, ctx.next_nt * BN + 8 * lane, p.V, nb);
    }
    Lse2 st;
    float zy = 0.0f;
    const float2 lg = make_float2(kLog2e, kLog2e);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = col_base + c * 32;
      if (col0 >= p.V) break;  // uniform across the warp
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      // the label's logit, in the one chunk that holds it (rarely any lane of a warp)
      if (static_cast<uint64_t>(ylocal - c * 32) < 32u)
        zy = pick32(v, ylocal, c * 32) +
             (bias != nullptr ? Elem<T>::load(bias + col_base + ylocal) : 0.0f);
      if (b2 != nullptr) {
        float t[32];
        const float4* bq = reinterpret_cast<const float4*>(b2 + c * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 bb = bq[k];
          const float2 t0 = __ffma2_rn(make_float2(v[4 * k], v[4 * k + 1]), lg,
                                       make_float2(bb.x, bb.y));
          const float2 t1 = __ffma2_rn(make_float2(v[4 * k + 2], v[4 * k + 3]), lg,
                                       make_float2(bb.z, bb.w));
          t[4 * k] = t0.x;
          t[4 * k + 1] = t0.y;
          t[4 * k + 2] = t1.x;
          t[4 * k + 3] = t1.y;
        }
        lse_add32_base2(t, p.V - col0, st);
      } else {
        lse_add32(v, p.V - col0, st);
      }
    }
    if (fetch_next) {  // the next tile's bias into the other half
      float* sn = reinterpret_cast<float*>(ctx.buf) + (ctx.aux ^ 1) * BN;
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 8; ++e) sn[8 * lane + e] = nb[e] * kLog2e;
      __syncwarp();
      ctx.aux ^= 1;
      ctx.aux_nt = ctx.next_nt;
    }
    if (row_ok && in_range(row, p.part_ld, p.status)) {
      p.part_m[nt * p.part_ld + row] = st.m;
      p.part_s[nt * p.part_ld + row] = st.s;
      if (ylocal >= 0 && ylocal < BN) p.zlab[row] = zy;
    }
  }
};

// Fused forward + backward, step 1: what EpiLse computes, and the tile's
// logits stored through TMA as u = z*log2(e) - m_tile (<= 0, in the input
// dtype) into the chunk buffer, so that the softmax can later be formed
// without recomputing the logits.  Storing the offset from the tile's own
// maximum keeps the rounding error of u small exactly where the softmax is
// large.  Two passes over the TMEM columns: the maximum first, then u and
// the sum of 2^u.
template <typename T>
struct EpiLseStore {
  using Params = typename EpiLse<T>::Params;
  template <int BN>
  __device__ static void tile(const Params& p, int mt, int nt, int row_in_tile, uint32_t taddr,
                              EpiCtx& ctx) {
    constexpr int CPS = 128 / static_cast<int>(sizeof(T));
    constexpr int EPV = Elem<T>::kPerVec;
    const int row = mt * kBM + row_in_tile;
    const bool row_ok = row < p.M;
    const int64_t y = row_ok ? p.labels[row] : -1;
    const int col_base = nt * BN;
    const int64_t ylocal = (y < 0) ? -1 : (y - p.v0) - col_base;
    const int r0 = mt * kBM + (row_in_tile & ~31);
    // pass 1: the tile maximum (the order of z equals the order of z*log2e)
    // and the label's logit, in the one chunk that holds it
    float mx = -INFINITY, zy = 0.0f;
    BiasAhead<T> bnext;
    if (p.bias != nullptr) bnext.fetch(p.bias, col_base, p.V);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = col_base + c * 32;
      if (col0 >= p.V) break;
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      if (p.bias != nullptr) {
        const BiasAhead<T> bcur = bnext;
        if (c + 1 < BN / 32) bnext.fetch(p.bias, col0 + 32, p.V);
        bcur.add(p.bias, col0, p.V, v);
      }
      if (static_cast<uint64_t>(ylocal - c * 32) < 32u) zy = pick32(v, ylocal, c * 32);
      if (col0 + 32 <= p.V) {
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, v[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < p.V) mx = fmaxf(mx, v[j]);
      }
    }
    const float m = mx * kLog2e;
    // pass 2: u = z*log2e - m by packed pairs, stored; the sum of 2^u in four
    // packed accumulators
    const float2 lg = make_float2(kLog2e, kLog2e), nm = make_float2(-m, -m);
    float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                     make_float2(0.0f, 0.0f)};
    if (p.bias != nullptr) bnext.fetch(p.bias, col_base, p.V);
#pragma unroll 1
    for (int g = 0; g < BN / CPS; ++g) {
      const int col0 = col_base + g * CPS;
      if (col0 >= p.V) break;
      uint4 packed[8];
#pragma unroll
      for (int h = 0; h < CPS / 32; ++h) {
        float v[32];
        tmem_ld32(taddr + g * CPS + h * 32, v);
        const int cb = col0 + h * 32;
        if (p.bias != nullptr) {
          const BiasAhead<T> bcur = bnext;
          if (cb + 32 < col_base + BN) bnext.fetch(p.bias, cb + 32, p.V);
          bcur.add(p.bias, cb, p.V, v);
        }
        const bool full = cb + 32 <= p.V;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float2 u = __ffma2_rn(make_float2(v[j], v[j + 1]), lg, nm);
          float2 e = make_float2(ex2(u.x), ex2(u.y));
          if (!full) {
            e.x = cb + j < p.V ? e.x : 0.0f;
            e.y = cb + j + 1 < p.V ? e.y : 0.0f;
          }
          acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], e);
          v[j] = u.x;
          v[j + 1] = u.y;
        }
#pragma unroll
        for (int k = 0; k < 32 / EPV; ++k) {
          float x[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[e] = v[k * EPV + e];
          packed[h * (32 / EPV) + k] = Elem<T>::pack(x);
        }
      }
      ctx.store_slab(packed, col0, r0, false);
    }
    const float2 a2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
    const float s = a2.x + a2.y;
    if (row_ok && in_range(row, p.part_ld, p.status)) {
      p.part_m[nt * p.part_ld + row] = m;
      p.part_s[nt * p.part_ld + row] = s;
      if (ylocal >= 0 && ylocal < BN) p.zlab[row] = zy;
    }
  }
};

// Backward step 1: dZ of one recomputed logits tile, stored as T through TMA
// (the output tensor map covers the chunk's [M, V] dZ buffer).
template <typename T>
struct EpiDlogits {
  struct Params {
    const void* bias;
    const int64_t* labels;  // chunk-relative (already offset)
    int64_t ignore_index;
    const float* lse;       // chunk-relative
    int reduction;
    int64_t num_label_tokens;
    const int64_t* n_valid;
    const float* grad_loss;
    int M, V;               // M = rows in this chunk; V = columns of this shard
    int64_t v0;             // vocabulary id of this shard's column 0
    int64_t V_total;        // vocabulary size (labels are checked against it)
    // bf16 only, or null: per 32-row group g of the chunk, the column sums of
    // the stored dZ at colsum[g * colsum_ld + column] (colsum_ld even), for
    // the bias gradient
    float* colsum = nullptr;
    int64_t colsum_ld = 0;
  };
  template <int BN>
  __device__ static void tile(const Params& p, int mt, int nt, int row_in_tile, uint32_t taddr,
                              EpiCtx& ctx) {
    tile_part<BN>(p, mt, nt, row_in_tile, taddr, ctx, 0, BN);
  }
  // Columns [c_lo, c_hi) of the tile (multiples of the 128-byte slab width):
  // with eight epilogue warps two warps share a TMEM lane quarter, each
  // forming and storing half of the tile's columns.
  template <int BN>
  __device__ static void tile_part(const Params& p, int mt, int nt, int row_in_tile,
                                   uint32_t taddr, EpiCtx& ctx, int c_lo, int c_hi) {
    constexpr int CPS = 128 / static_cast<int>(sizeof(T));  // columns per 128-byte row slab
    constexpr int EPV = Elem<T>::kPerVec;
    const int row = mt * kBM + row_in_tile;
    const bool row_ok = row < p.M;
    const int64_t y = row_ok ? p.labels[row] : p.ignore_index;
    const bool valid = row_ok && y != p.ignore_index && label_ok(y, p.V_total);
    const float c = valid ? grad_coef(p.reduction, p.num_label_tokens, p.n_valid, p.grad_loss)
                          : 0.0f;
    const float lse2 = row_ok ? p.lse[row] * kLog2e : 0.0f;
    // c * 2^(t - lse2) = sign(c) * 2^(t - (lse2 - log2|c|)): one FFMA and one
    // ex2 per element; a negative c flips the sign bits of the packed words
    const float l2c = c != 0.0f ? lse2 - log2f(fabsf(c)) : 0.0f;
    const uint32_t neg = c < 0.0f ? (sizeof(T) == 2 ? 0x80008000u : 0x80000000u) : 0u;
    const float2 lg = make_float2(kLog2e, kLog2e), nl = make_float2(-l2c, -l2c);
    const int col_base = nt * BN;
    const int64_t ylocal = valid ? (y - p.v0) - col_base : -1;
    const int r0 = mt * kBM + (row_in_tile & ~31);
    BiasAhead<T> bnext;
    if (p.bias != nullptr) bnext.fetch(p.bias, col_base + c_lo, p.V);
#pragma unroll 1
    for (int g = c_lo / CPS; g < c_hi / CPS; ++g) {
      const int col0 = col_base + g * CPS;
      if (col0 >= p.V) break;  // uniform across the warp
      uint4 packed[8];
#pragma unroll
      for (int h = 0; h < CPS / 32; ++h) {
        float v[32];
        tmem_ld32(taddr + g * CPS + h * 32, v);
        const int cl = g * CPS + h * 32;  // column within the tile
        if (p.bias != nullptr) {
          const BiasAhead<T> bcur = bnext;
          if (cl + 32 < c_hi) bnext.fetch(p.bias, col_base + cl + 32, p.V);
          bcur.add(p.bias, col_base + cl, p.V, v);
        }
        if (c == 0.0f) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.0f;
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 t = __ffma2_rn(make_float2(v[j], v[j + 1]), lg, nl);
            v[j] = ex2(t.x);
            v[j + 1] = ex2(t.y);
          }
        }
        const bool has_label = static_cast<uint64_t>(ylocal - cl) < 32u;
        if (has_label) {  // the one-hot term, in the chunk holding the label
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = neg ? -v[j] : v[j];
            if (cl + j == ylocal) v[j] -= c;
          }
        }
#pragma unroll
        for (int k = 0; k < 32 / EPV; ++k) {
          float x[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[e] = v[k * EPV + e];
          uint4 w = Elem<T>::pack(x);
          if (!has_label) {
            w.x ^= neg;
            w.y ^= neg;
            w.z ^= neg;
            w.w ^= neg;
          }
          packed[h * (32 / EPV) + k] = w;
        }
      }
      ctx.store_slab(packed, col0, r0, false);
      if constexpr (sizeof(T) == 2) {
        if (p.colsum != nullptr) {  // this warp's 32 rows of the slab, summed
          const float2 cs = ctx.last_slab_bf16_column_sums();
          const int col = col0 + 2 * (row_in_tile & 31);
          float* dst = p.colsum + static_cast<int64_t>(r0 >> 5) * p.colsum_ld + col;
          if (col + 1 < p.V)
            *reinterpret_cast<float2*>(dst) = cs;
          else if (col < p.V)
            dst[0] = cs.x;
        }
      }
    }
  }
};

// Stores the accumulator as OutT through TMA (grad_H), or, with kAccumulate and
// beta = 1, adds it into the existing fp32 output with a TMA reduce-add
// (grad_W): the read-modify-write happens in L2, not on the SM.
template <typename OutT, bool kAccumulate>
struct EpiStore {
  struct Params {
    int M, N;
    int beta;  // accumulate variant: 1 adds to the existing contents
  };
  template <int BN>
  __device__ static void tile(const Params& p, int mt, int nt, int row_in_tile, uint32_t taddr,
                              EpiCtx& ctx) {
    constexpr int CPS = 128 / static_cast<int>(sizeof(OutT));
    constexpr int EPV = Elem<OutT>::kPerVec;
    const int r0 = mt * kBM + (row_in_tile & ~31);
    const bool reduce = kAccumulate && p.beta != 0;
#pragma unroll 1
    for (int g = 0; g < BN / CPS; ++g) {
      const int col0 = nt * BN + g * CPS;
      if (col0 >= p.N) break;
      uint4 packed[8];
#pragma unroll
      for (int h = 0; h < CPS / 32; ++h) {
        float v[32];
        tmem_ld32(taddr + g * CPS + h * 32, v);
#pragma unroll
        for (int k = 0; k < 32 / EPV; ++k) {
          float x[EPV];
#pragma unroll
          for (int e = 0; e < EPV; ++e) x[e] = v[k * EPV + e];
          packed[h * (32 / EPV) + k] = Elem<OutT>::pack(x);
        }
      }
      ctx.store_slab(packed, col0, r0, reduce);
    }
  }
};

// ------------------------------------------------------------ small kernels

// Merge of the per-(row, vocab tile) partials of 32 rows per block of nw
// warps (nw = min(16, tiles)): warp w merges the tiles p = w, w + nw, ... of
// its lane's row (lane = row, so each load of a warp reads 32 consecutive rows
// of one tile: 128 bytes), then warp 0 merges the nw warp states of each row in
// warp order.  Fixed order, so the result is the same on every run.
constexpr int kCombineRows = 32;
constexpr int kCombineWarps = 16;

static unsigned combine_threads(int nparts) {
  return static_cast<unsigned>(32 * std::max(1, std::min(kCombineWarps, nparts)));
}

__device__ __forceinline__ bool combine_rows(const float* __restrict__ part_m,
                                             const float* __restrict__ part_s, int nparts,
                                             int64_t part_ld, int64_t N, int64_t& row,
                                             Lse2& all) {
  __shared__ float sm[kCombineWarps][kCombineRows], ss[kCombineWarps][kCombineRows];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  row = static_cast<int64_t>(blockIdx.x) * kCombineRows + lane;
  Lse2 st;
  if (row < N) {
#pragma unroll 4
    for (int p = warp; p < nparts; p += nw)
      st.merge(part_m[p * part_ld + row], part_s[p * part_ld + row]);
  }
  sm[warp][lane] = st.m;
  ss[warp][lane] = st.s;
  __syncthreads();
  if (warp != 0 || row >= N) return false;
  for (int w = 0; w < nw; ++w) all.merge(sm[w][lane], ss[w][lane]);
  return true;
}

// Forward: per row, the tile partials merged into the lse, and the row loss
// from the label logit (the tile holding the label wrote it).
__global__ void __launch_bounds__(kCombineRows * kCombineWarps) lse_combine_kernel(
    const float* __restrict__ part_m, const float* __restrict__ part_s, int nparts,
    int64_t part_ld, const float* __restrict__ zlab, const int64_t* __restrict__ labels,
    int64_t N, int64_t V, int64_t ignore_index, float* __restrict__ lse_out,
    float* __restrict__ loss_rows, float* __restrict__ label_logit, int32_t* status) {
  int64_t row;
  Lse2 st;
  if (!combine_rows(part_m, part_s, nparts, part_ld, N, row, st)) return;
  const float lse = st.m * kLn2 + logf(st.s);
  lse_out[row] = lse;
  const int64_t y = labels[row];
  float li = 0.0f, zy = NAN;
  if (y != ignore_index) {
    if (label_ok(y, V)) {
      zy = zlab[row];
      li = lse - zy;
    } else {
      set_status(status, FLCE_ELABEL);
    }
  }
  loss_rows[row] = li;
  if (label_logit != nullptr) label_logit[row] = zy;
}

// Vocabulary-parallel forward: merges this shard's tile partials of each row
// into (m, s) (base-2 max and sum over the shard's columns) and the label logit
// when the label lies in the shard (0 otherwise).
__global__ void __launch_bounds__(kCombineRows * kCombineWarps) shard_combine_kernel(
    const float* __restrict__ part_m, const float* __restrict__ part_s, int nparts,
    int64_t part_ld, const float* __restrict__ zlab, const int64_t* __restrict__ labels,
    int64_t N, int64_t V_shard, int64_t v0, int64_t ignore_index, float* __restrict__ m_out,
    float* __restrict__ s_out, float* __restrict__ zy_out) {
  int64_t row;
  Lse2 st;
  if (!combine_rows(part_m, part_s, nparts, part_ld, N, row, st)) return;
  m_out[row] = st.m;
  s_out[row] = st.s;
  const int64_t y = labels[row];
  const bool in_shard = y != ignore_index && y >= v0 && y < v0 + V_shard;
  zy_out[row] = in_shard ? zlab[row] : 0.0f;
}

// s_scaled = s * 2^(m - m_global): a shard's sum expressed relative to the
// maximum over all shards (0 when the shard's maximum is -inf).
__global__ void __launch_bounds__(256) shard_rescale_kernel(const float* __restrict__ m,
                                                            const float* __restrict__ s,
                                                            const float* __restrict__ m_global,
                                                            int64_t N, float* __restrict__ out) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  out[i] = (m[i] == -INFINITY) ? 0.0f : s[i] * ex2(m[i] - m_global[i]);
}

// lse = (M + log2 S) ln 2 from the global (M, S); loss_i = valid (lse - z_y).
__global__ void __launch_bounds__(256) shard_finish_kernel(
    const float* __restrict__ m_global, const float* __restrict__ s_global,
    const float* __restrict__ zy_global, const int64_t* __restrict__ labels, int64_t N,
    int64_t V_total, int64_t ignore_index, float* __restrict__ lse_out,
    float* __restrict__ loss_rows, int32_t* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const float lse = m_global[i] * kLn2 + logf(s_global[i]);
  lse_out[i] = lse;
  const int64_t y = labels[i];
  float li = 0.0f;
  if (y != ignore_index) {
    if (label_ok(y, V_total))
      li = lse - zy_global[i];
    else
      set_status(status, FLCE_ELABEL);
  }
  loss_rows[i] = li;
}

constexpr int kColSplits = 32;

// Rows of partial column sums the eight-warp dZ epilogue writes for a chunk
// of C rows (one per 32 rows of its 128-row tiles); 0 where it cannot run.
static int64_t dz_colsum_rows(int dt, int64_t D, int64_t C) {
  return dt == FLCE_BF16 && D <= 1024 ? (C + kBM - 1) / kBM * (kBM / 32) : 0;
}

// Column sums of dZ [M, ldd] over row slices: part[s, v] = sum of rows in slice
// s.  Each thread sums one 16-byte vector of columns (the chunk buffer's row
// stride is a multiple of 64 elements and its start 256-byte aligned, so every
// vector lies inside the allocation; columns at or past V are not written).
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial_kernel(const T* __restrict__ dz, int M,
                                                             int64_t ldd, int V,
                                                             float* __restrict__ part) {
  constexpr int EPV = Elem<T>::kPerVec;
  const int v0 = (blockIdx.x * blockDim.x + threadIdx.x) * EPV;
  if (v0 >= V) return;
  const int s = blockIdx.y;
  const int per = (M + kColSplits - 1) / kColSplits;
  const int r0 = s * per, r1 = min(M, r0 + per);
  float acc[EPV];
#pragma unroll
  for (int e = 0; e < EPV; ++e) acc[e] = 0.0f;
  const uint4* q = reinterpret_cast<const uint4*>(dz + static_cast<int64_t>(r0) * ldd + v0);
  const int64_t step = ldd / EPV;
#pragma unroll 8
  for (int r = r0; r < r1; ++r, q += step) {
    float x[EPV];
    Elem<T>::unpack(__ldcs(q), x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) acc[e] += x[e];
  }
#pragma unroll
  for (int e = 0; e < EPV; ++e)
    if (v0 + e < V) part[static_cast<int64_t>(s) * V + v0 + e] = acc[e];
}

// out[v] (+)= the sum of the nparts partial column sums part[s * ld + v].  A
// block takes 32 columns: warp w sums the partials s = w, w + 8, ... in order
// (each load of a warp reads 32 consecutive columns), then the eight warp sums
// are added in warp order, so the result is the same on every run.
constexpr int kColFinalWarps = 8;

__global__ void __launch_bounds__(32 * kColFinalWarps) colsum_final_kernel(
    const float* __restrict__ part, int nparts, int64_t ld, int V, float* __restrict__ out,
    int beta) {
  __shared__ float red[kColFinalWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int v = blockIdx.x * 32 + lane;
  float acc = 0.0f;
  if (v < V) {
#pragma unroll 4
    for (int s = warp; s < nparts; s += kColFinalWarps) acc += part[static_cast<int64_t>(s) * ld + v];
  }
  red[warp][lane] = acc;
  __syncthreads();
  if (warp != 0 || v >= V) return;
  float total = beta ? out[v] : 0.0f;
  for (int w = 0; w < kColFinalWarps; ++w) total += red[w][lane];
  out[v] = total;
}

// out[c, r] = in[r, c] for a [R, Cc] matrix of 4-byte elements (32 x 32 tiles
// through shared memory; both sides coalesced).  The tf32 tensor-core path
// takes only K-major operands, so the fp32 backward transposes its MN-major
// operands with this kernel.
__global__ void __launch_bounds__(256) transpose32_kernel(const float* __restrict__ in, int R,
                                                          int Cc, int64_t ld_in,
                                                          float* __restrict__ out,
                                                          int64_t ld_out) {
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int k = ty; k < 32; k += 8) {
    const int r = r0 + k, c = c0 + tx;
    if (r < R && c < Cc) tile[k][tx] = in[static_cast<int64_t>(r) * ld_in + c];
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int c = c0 + k, r = r0 + tx;
    if (c < Cc && r < R) out[static_cast<int64_t>(c) * ld_out + r] = tile[tx][k];
  }
}

static void transpose32(const float* in, int R, int Cc, int64_t ld_in, float* out,
                        int64_t ld_out, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((Cc + 31) / 32), static_cast<unsigned>((R + 31) / 32));
  transpose32_kernel<<<grid, 256, 0, s>>>(in, R, Cc, ld_in, out, ld_out);
}

// Fused forward + backward, step 3: in place over the chunk buffer,
// dZ = (2^(u + m_tile - lse*log2(e)) - [j == y]) * coef, one CTA per row
// (grid-stride); the row's per-tile maxima are staged in shared memory first.
constexpr int kMaxTilesPerRow = 8192;  // V < 2^21 with 256-wide tiles

template <typename T>
__global__ void __launch_bounds__(256) dz_from_u_kernel(
    T* buf, int C, int V, int64_t ldd, const float* __restrict__ part_m, int nparts,
    int64_t part_ld, const float* __restrict__ lse, const int64_t* __restrict__ labels,
    int64_t ignore_index, int reduction, int64_t num_label_tokens, const int64_t* n_valid,
    const float* grad_loss) {
  constexpr int EPV = Elem<T>::kPerVec;
  extern __shared__ float mrow[];
  const float coef = grad_coef(reduction, num_label_tokens, n_valid, grad_loss);
  const int nvec = V / EPV;
  for (int row = blockIdx.x; row < C; row += gridDim.x) {
    const int64_t y = labels[row];
    const bool valid = (y != ignore_index) && label_ok(y, V);
    const float c = valid ? coef : 0.0f;
    const float lse2 = lse[row] * kLog2e;
    __syncthreads();  // mrow of the previous row fully used
    for (int t = threadIdx.x; t < nparts; t += blockDim.x)
      mrow[t] = part_m[static_cast<int64_t>(t) * part_ld + row] - lse2;
    __syncthreads();
    T* r = buf + static_cast<int64_t>(row) * ldd;
    uint4* rv = reinterpret_cast<uint4*>(r);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float x[EPV];
      const int j0 = v * EPV;
      if (c == 0.0f) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) x[e] = 0.0f;
      } else {
        Elem<T>::unpack(rv[v], x);
        const float off = mrow[j0 >> 8];  // all EPV columns lie in one 256-wide tile
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          x[e] = (ex2(x[e] + off) - (j0 + e == y ? 1.0f : 0.0f)) * c;
      }
      rv[v] = Elem<T>::pack(x);
    }
    for (int j = nvec * EPV + threadIdx.x; j < V; j += blockDim.x) {
      float d = 0.0f;
      if (c != 0.0f)
        d = (ex2(Elem<T>::load(r + j) + mrow[j >> 8]) - (j == y ? 1.0f : 0.0f)) * c;
      Elem<T>::store(r + j, d);
    }
  }
}

// n_valid = number of labels that are not ignore_index and lie in [0, V).
__global__ void __launch_bounds__(1024) count_valid_kernel(const int64_t* __restrict__ labels,
                                                           int64_t N, int64_t V,
                                                           int64_t ignore_index,
                                                           int64_t* __restrict__ n_valid) {
  __shared__ long long sc[1024];
  long long cnt = 0;
  for (int64_t i = threadIdx.x; i < N; i += 1024) {
    const int64_t y = labels[i];
    cnt += (y != ignore_index && label_ok(y, V)) ? 1 : 0;
  }
  sc[threadIdx.x] = cnt;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) sc[threadIdx.x] += sc[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *n_valid = sc[0];
}

// x *= g (one float read per thread; nothing is written when g == 1).
template <typename T>
__global__ void __launch_bounds__(256) scale_kernel(T* x, int64_t n, const float* g) {
  const float s = *g;
  if (s == 1.0f) return;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    Elem<T>::store(x + i, Elem<T>::load(x + i) * s);
}

// x[0..n) = 0: the weight and bias gradients of an empty batch.
__global__ void __launch_bounds__(256) zero_kernel(float* x, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = 0.0f;
}

static int launch_zero(float* x, int64_t n, cudaStream_t s) {
  if (x == nullptr || n == 0) return FLCE_OK;
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, sm_count() * 8));
  zero_kernel<<<grid, 256, 0, s>>>(x, n);
  return launch_status("zero_kernel launch");
}

// Backward of an empty batch (N = 0): the loss has no terms, so grad_W (unless
// accumulated) and grad_bias are zero; grad_H has no rows.
static int empty_bwd(int64_t D, int64_t V, float* grad_W, int accumulate_grad_W,
                     float* grad_bias, cudaStream_t s) {
  int rc = accumulate_grad_W ? FLCE_OK : launch_zero(grad_W, V * D, s);
  if (rc != FLCE_OK) return rc;
  return launch_zero(grad_bias, V, s);
}

// out[r, d] = sum over s of part[s * split_stride + r * D + d], in split order
// (deterministic), converted to OutT.  Closes a split-K contraction.
// Four consecutive elements per thread and step (16-byte loads of each split;
// C x D is a multiple of 4 since D * sizeof(input) is a multiple of 16, and
// part, split_stride and out are aligned to match).
template <typename OutT>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ part,
                                                            int S, int64_t split_stride, int C,
                                                            int D, OutT* __restrict__ out) {
  const int64_t n4 = static_cast<int64_t>(C) * D / 4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int sp = 0; sp < S; ++sp) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(part + sp * split_stride) + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4*>(out)[i] = acc;
    } else {
      reinterpret_cast<uint2*>(out)[i] =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

// --------------------------------------------------------------- host: TMA

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// cuTensorMapEncodeTiled is a driver call and needs a current context on the
// calling thread.  A thread that has only launched kernels through a runtime
// may have none bound yet (e.g. an autograd worker thread): then bind the
// current device's primary context.  A thread that has one is left alone (so
// nothing but a query runs while a stream is being captured).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

static int bind_context() {
  CtxGetCurrentFn get = ctx_get_current_fn();
  if (get != nullptr) {
    CUcontext ctx = nullptr;
    if (get(&ctx) == CUDA_SUCCESS && ctx != nullptr) return FLCE_OK;
  }
  int dev = 0;
  int rc = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc != FLCE_OK) return rc;
  return cuda_status(cudaSetDevice(dev), "cudaSetDevice");
}

// 2-D map over a row-major matrix [outer, inner] with the given row stride, box
// {128 bytes of inner, box_outer rows}, 128-byte swizzle, zero fill outside.
static int make_map(CUtensorMap* m, const void* base, int dt, uint64_t inner, uint64_t outer,
                    uint64_t row_stride_elems, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) {
    record_cuda_error(cudaErrorUnknown, "cuTensorMapEncodeTiled entry point");
    return FLCE_ECUDA;
  }
  const uint64_t es = dtype_size(dt);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_elems * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt == FLCE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "cuTensorMapEncodeTiled CUresult=%d addr=%p dims={%llu,%llu} stride=%llu "
             "box={%u,%u} map@%p",
             static_cast<int>(r), base, static_cast<unsigned long long>(inner),
             static_cast<unsigned long long>(outer),
             static_cast<unsigned long long>(row_stride_elems * es), box[0], box[1],
             static_cast<void*>(m));
    record_cuda_error(cudaErrorUnknown, msg);
    return FLCE_ECUDA;
  }
  return FLCE_OK;
}

// Operand description for the host launcher.
struct Operand {
  const void* ptr;
  int64_t rows;      // extent along M (for A) or N (for B)
  int64_t k;         // extent along K
  int64_t ld;        // row stride in elements of the stored matrix
  bool mn_major;     // stored as [K, rows] (true) or [rows, K] (false)
};

static int make_operand_map(CUtensorMap* m, const Operand& op, int dt, int tile_rows) {
  const int ek = 128 / static_cast<int>(dtype_size(dt));
  if (!op.mn_major) return make_map(m, op.ptr, dt, op.k, op.rows, op.ld, tile_rows);
  return make_map(m, op.ptr, dt, op.rows, op.k, op.ld, ek);
}

// Per-device, per-kernel host state: whether the dynamic shared-memory limit
// has been raised, and the number of resident CTA pairs.  Filled on the first
// launch of each kernel on each device (ids < 64), so that later launches -
// including launches inside a stream capture - only enqueue work.
static std::mutex g_attr_mutex;
static std::vector<std::pair<const void*, int>> g_attr_done;  // (kernel, device)

template <typename Kern>
static int raise_smem_once(Kern kern, int bytes, const char* what) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const void* key = reinterpret_cast<const void*>(kern);
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  for (const auto& e : g_attr_done)
    if (e.first == key && e.second == dev) return FLCE_OK;
  const int rc = cuda_status(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), what);
  if (rc == FLCE_OK) g_attr_done.emplace_back(key, dev);
  return rc;
}

// Output of an epilogue that stores through TMA: row-major [rows, cols] with
// row stride ld (elements), written in boxes of 32 rows x 128 bytes.
struct OutDesc {
  void* ptr;
  int dt;
  int64_t rows, cols, ld;
};

// Which bf16 contractions run on CTA pairs (tc_gemm_pair_kernel) instead of one
// CTA per tile: a bit mask of GemmRole.
// kWideDz (not a contraction): the dZ contraction at K <= 1024 runs on one CTA
// per tile with eight epilogue warps instead (launch_dz_gemm).
enum GemmRole : int { kRoleFwd = 1, kRoleDz = 2, kRoleGradH = 4, kRoleGradW = 8, kRoleRaw = 16 };
constexpr int kWideDz = 32;
static std::atomic<int> g_pair_mask{kRoleDz | kRoleGradW | kRoleRaw | kWideDz};

template <int BN, bool A_MN, bool B_MN, class Epi>
static int launch_gemm_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                            int M, int N, int K, int group_m, const typename Epi::Params& ep,
                            int32_t* status, cudaStream_t s, const EpiPre& pre) {
  using G = PairGeo<BN>;
  GemmArgs ga;
  ga.M = M;
  ga.N = N;
  ga.K = K;
  ga.nMt = (M + 2 * kBM - 1) / (2 * kBM);
  ga.nNt = (N + BN - 1) / BN;
  ga.nK = (K + G::kEK - 1) / G::kEK;
  ga.group_m = std::max(1, std::min((group_m + 1) / 2, ga.nMt));
  ga.status = status;
  ga.k_splits = 1;
  ga.kb_per_split = ga.nK;
  ga.pre = pre;
  const int tiles = ga.nMt * ga.nNt;
  if (tiles == 0) return pre.kind != 0 ? FLCE_EINVAL : FLCE_OK;  // the work would be lost
  auto kern = tc_gemm_pair_kernel<BN, A_MN, B_MN, Epi>;
  int rc = raise_smem_once(kern, G::kSmemBytes, "cudaFuncSetAttribute(tc_gemm_pair_kernel)");
  if (rc != FLCE_OK) return rc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many pairs as can be resident at once (on GB300 all 152 SMs pair up: 76)
  static std::atomic<int> pairs_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  int max_pairs = pairs_cache[dev & 63].load();
  if (max_pairs <= 0) {
    cfg.gridDim = dim3(2 * static_cast<unsigned>(std::min(tiles, sm_count() / 2)), 1, 1);
    rc = cuda_status(cudaOccupancyMaxActiveClusters(&max_pairs, kern, &cfg),
                     "cudaOccupancyMaxActiveClusters");
    if (rc != FLCE_OK) return rc;
    if (max_pairs < 1) return FLCE_ENOSUP;
    pairs_cache[dev & 63].store(max_pairs);
  }
  cfg.gridDim = dim3(2 * static_cast<unsigned>(std::min(tiles, max_pairs)), 1, 1);
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, ga, ep),
                     "cudaLaunchKernelEx(tc_gemm_pair_kernel)");
}

// pre: work for the epilogue warps before their first tile (EpiPre).
template <typename T, int BN, bool A_MN, bool B_MN, class Epi, int EW = 4>
static int launch_gemm(int role, const Operand& a, const Operand& b, const OutDesc* out, int M,
                       int N, int K, int group_m, const typename Epi::Params& ep,
                       int32_t* status, cudaStream_t s, int k_splits = 1,
                       const EpiPre& pre = EpiPre()) {
  using G = GemmGeo<T, BN, EW>;
  const int dt = sizeof(T) == 2 ? FLCE_BF16 : FLCE_F32;
  CUtensorMap ma, mb, mc;
  const bool pair = EW == 4 && sizeof(T) == 2 && BN == 256 && k_splits == 1 &&
                    (g_pair_mask.load() & role) != 0;
  int rc = make_operand_map(&ma, a, dt, kBM);
  if (rc != FLCE_OK) return rc;
  rc = make_operand_map(&mb, b, dt, pair ? BN / 2 : BN);
  if (rc != FLCE_OK) return rc;
  if (out != nullptr) {
    rc = make_map(&mc, out->ptr, out->dt, out->cols, out->rows, out->ld, 32);
    if (rc != FLCE_OK) return rc;
  } else {
    mc = ma;  // unused by epilogues that do not store through TMA
  }
  if constexpr (sizeof(T) == 2 && BN == 256 && EW == 4) {
    if (pair) return launch_gemm_pair<BN, A_MN, B_MN, Epi>(ma, mb, mc, M, N, K, group_m, ep,
                                                         status, s, pre);
  }
  GemmArgs ga;
  ga.M = M;
  ga.N = N;
  ga.K = K;
  ga.nMt = (M + kBM - 1) / kBM;
  ga.nNt = (N + BN - 1) / BN;
  ga.nK = (K + G::kEK - 1) / G::kEK;
  ga.k_splits = std::max(1, std::min(k_splits, ga.nK));
  ga.kb_per_split = (ga.nK + ga.k_splits - 1) / ga.k_splits;
  ga.k_splits = (ga.nK + ga.kb_per_split - 1) / ga.kb_per_split;  // no empty split
  ga.group_m = std::max(1, std::min(group_m, ga.nMt * ga.k_splits));
  ga.status = status;
  ga.pre = pre;
  const int tiles = ga.nMt * ga.k_splits * ga.nNt;
  if (tiles == 0) return pre.kind != 0 ? FLCE_EINVAL : FLCE_OK;  // the work would be lost
  auto kern = tc_gemm_kernel<T, BN, A_MN, B_MN, Epi, EW>;
  rc = raise_smem_once(kern, G::kSmemBytes, "cudaFuncSetAttribute(tc_gemm_kernel)");
  if (rc != FLCE_OK) return rc;
  const int grid = std::min(tiles, sm_count());
  kern<<<grid, G::kThreads, G::kSmemBytes, s>>>(ma, mb, mc, ga, ep);
  return launch_status("tc_gemm_kernel launch");
}

// Group of M-tiles sharing one sweep over the N-tiles: as many 128-row slabs of
// the A operand as fit in about 40 MB of L2.
static int group_for(int64_t K, int dt, int nMt) {
  const int64_t slab = static_cast<int64_t>(kBM) * K * static_cast<int64_t>(dtype_size(dt));
  int64_t g = (40ll << 20) / std::max<int64_t>(slab, 1);
  g = std::max<int64_t>(1, std::min<int64_t>(g, nMt));
  return static_cast<int>(g);
}

// Number of K splits launch_gemm really uses for `requested` (no empty split).
static int effective_splits(int nK, int requested) {
  int S = std::max(1, std::min(requested, nK));
  const int per = (nK + S - 1) / S;
  return (nK + per - 1) / per;
}

// grad_H of a C-row chunk has only ceil(C/128) * ceil(D/256) output tiles; when
// they cannot fill half of the SMs, its long K (= V) is split so that they do.
static int grad_h_splits(int64_t C, int64_t D, int64_t V, int dt) {
  const int64_t tiles = ((C + kBM - 1) / kBM) * ((D + 255) / 256);
  const int64_t sms = sm_count();
  if (tiles * 2 > sms) return 1;
  const int nK = static_cast<int>((V + (128 / dtype_size(dt)) - 1) / (128 / dtype_size(dt)));
  int64_t S = std::min<int64_t>(sms / tiles, 8);
  S = std::min<int64_t>(S, nK / 16);
  return effective_splits(nK, static_cast<int>(std::max<int64_t>(S, 1)));
}

// ------------------------------------------------------------ workspace plan

constexpr int kBNFwd = 256;

struct FlcePlan {
  int64_t ldV;         // row stride of the dZ chunk buffer (elements)
  int64_t chunk;
  int nparts;          // vocab tiles of the forward
  int64_t part_ld;
  size_t off_part_m, off_part_s, off_zlab, off_rows, fwd_bytes;
  size_t off_dz, off_colsum, off_hpart, bwd_bytes;
  // fp32 only: K-major copies of the operands the tf32 MMA cannot read MN-major
  int64_t ldVt, ldCt;
  size_t off_Wt, off_dzT, off_HT;
  // fused forward + backward: chunk-sized partials after the backward buffers
  int64_t fpart_ld;
  size_t off_fpart_m, off_fpart_s, off_fzlab, off_frows, fused_bytes;
  size_t total;
  // vocabulary slices (vchunk > 0): the backward runs over all rows at once,
  // slice by slice of vchunk columns; dZ of a slice is [N, ldVc], and grad_H
  // accumulates in fp32 at off_hacc ([N, D]) before one rounding
  int64_t vchunk = 0, ldVc = 0;
  size_t off_hacc = 0;
};

static FlcePlan plan(int dt, int64_t N, int64_t D, int64_t V, int64_t chunk,
                     bool bwd_split = false);

// Bytes of extra device memory the default chunk may use: one [2048, V] fp32
// tile.  Automodel PR #2996 ("Motivation") bounds the fp32 transient of its
// chunked loss by chunk_size x V x 4 bytes whatever the sequence length; the
// chunk of that bound is fixed here at 2048 rows.
static size_t extra_memory_budget(int64_t V) { return static_cast<size_t>(2048) * V * 4; }

// Rows per backward chunk.  The largest multiple of 128 rows (at most 4864)
// whose workspace, for flce_bwd and for flce_fwd_bwd alike, stays within the
// budget above (the dZ chunk buffer of C x ldV input elements dominates it)
// is the cap; within [cap/2, cap], C is chosen so that the grad_H contraction,
// whose tile count C/128 x D/256 is the smallest of the backward's, fills
// whole waves of the GPU's SMs over all chunks of N (the largest such C).
// fp32 inputs also keep transposed operands of D x V floats, which the
// budget cannot hold at large sizes: their cap falls to 128 rows.
static int64_t default_chunk(int dt, int64_t N, int64_t D, int64_t V) {
  const int64_t n128 = (N + 127) / 128 * 128;
  const size_t budget = extra_memory_budget(V);
  int64_t cap = std::min<int64_t>(4864, n128);
  while (cap > 128 && plan(dt, N, D, V, cap).fused_bytes > budget) cap -= 128;
  if (n128 <= cap) return n128;
  const int64_t sms = sm_count();
  const int64_t nNt = (D + 255) / 256;
  int64_t best = cap;
  double best_eff = -1.0;
  for (int64_t c = cap; c >= std::max<int64_t>(128, cap / 2); c -= 128) {
    int64_t tiles = 0, slots = 0;
    for (int64_t r0 = 0; r0 < N; r0 += c) {
      const int64_t t = (std::min(c, N - r0) + 127) / 128 * nNt;
      tiles += t;
      slots += (t + sms - 1) / sms * sms;
    }
    const double eff = static_cast<double>(tiles) / static_cast<double>(slots);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = c;
    }
  }
  return best;
}

// The backward's split: chunk > 0, row chunks of that many rows; chunk == 0,
// default_chunk; chunk < 0 (flce_bwd only, bwd_split set; bf16), vocabulary
// slices of -chunk columns.  A slice runs over all N rows, so grad_W is
// written once (row chunks read and write the fp32 grad_W once more per
// chunk after the first) and grad_H accumulates in an fp32 [N, D] buffer
// instead (one rounding to the input dtype at the end).  At N=8192 D=4096
// V=128256, three slices of 42752 columns move 0.9 GB of accumulator bytes
// where three row chunks move 10.5 GB, yet the step was only 0.3% faster
// (21.48 against 21.55 ms, one box), and grad_W is then one fp32 sweep over
// all N rows in the tensor core, whose accumulation rounding grows with the
// sweep (row chunks add their partial sums in L2, rounding to nearest): the
// default stays with rows.
static FlcePlan plan(int dt, int64_t N, int64_t D, int64_t V, int64_t chunk, bool bwd_split) {
  FlcePlan p;
  const size_t es = dtype_size(dt);
  if (chunk < 0 && !bwd_split) chunk = 0;
  if (chunk < 0) {
    p.vchunk = std::min<int64_t>(-chunk, V);
    p.ldVc = (p.vchunk + 63) / 64 * 64;
    chunk = N;
  }
  p.chunk = chunk > 0 ? chunk : default_chunk(dt, N, D, V);
  p.ldV = (V + 63) / 64 * 64;
  p.nparts = static_cast<int>((V + kBNFwd - 1) / kBNFwd);
  p.part_ld = (N + 63) / 64 * 64;
  size_t o = 0;
  p.off_part_m = o;
  o += round_up(static_cast<size_t>(p.nparts) * p.part_ld * 4, 256);
  p.off_part_s = o;
  o += round_up(static_cast<size_t>(p.nparts) * p.part_ld * 4, 256);
  p.off_zlab = o;
  o += round_up(static_cast<size_t>(N) * 4, 256);
  p.off_rows = o;
  o += round_up(static_cast<size_t>(N) * 4, 256);
  p.fwd_bytes = o;
  o = 0;
  p.off_dz = o;
  o += round_up(static_cast<size_t>(std::min<int64_t>(p.chunk, N)) * p.ldV * es, 256);
  p.off_colsum = o;
  o += round_up(std::max(static_cast<size_t>(kColSplits) * V,
                         static_cast<size_t>(dz_colsum_rows(dt, D, std::min<int64_t>(p.chunk, N))) *
                             p.ldV) *
                    4,
                256);
  {
    // split-K partials of grad_H, for the full chunk and for the last one
    const int64_t c1 = std::min<int64_t>(p.chunk, N);
    const int64_t c2 = N % p.chunk == 0 ? c1 : N % p.chunk;
    size_t need = 0;
    for (int64_t c : {c1, c2}) {
      const int S = grad_h_splits(c, D, V, dt);
      if (S > 1)
        need = std::max(need, static_cast<size_t>(S) * ((c + kBM - 1) / kBM) * kBM * D * 4);
    }
    p.off_hpart = o;
    o += round_up(need, 256);
  }
  p.ldVt = (V + 3) / 4 * 4;
  p.ldCt = (std::min<int64_t>(p.chunk, N) + 3) / 4 * 4;
  p.off_Wt = p.off_dzT = p.off_HT = 0;
  if (dt == FLCE_F32) {
    p.off_Wt = o;
    o += round_up(static_cast<size_t>(D) * p.ldVt * 4, 256);
    p.off_dzT = o;
    o += round_up(static_cast<size_t>(V) * p.ldCt * 4, 256);
    p.off_HT = o;
    o += round_up(static_cast<size_t>(D) * p.ldCt * 4, 256);
  }
  if (p.vchunk > 0) {
    o = 0;
    p.off_dz = o;
    o += round_up(static_cast<size_t>(N) * p.ldVc * es, 256);
    p.off_colsum = o;
    o += round_up(std::max(static_cast<size_t>(kColSplits) * p.vchunk,
                           static_cast<size_t>(dz_colsum_rows(dt, D, N)) * p.ldVc) *
                      4,
                  256);
    p.off_hpart = o;
    p.off_hacc = o;
    o += round_up(static_cast<size_t>(N) * D * 4, 256);
  }
  p.bwd_bytes = o;
  p.total = std::max(p.fwd_bytes, p.bwd_bytes);
  p.fpart_ld = (std::min<int64_t>(p.chunk, N) + 63) / 64 * 64;
  p.off_fpart_m = o;
  o += round_up(static_cast<size_t>(p.nparts) * p.fpart_ld * 4, 256);
  p.off_fpart_s = o;
  o += round_up(static_cast<size_t>(p.nparts) * p.fpart_ld * 4, 256);
  p.off_fzlab = o;
  o += round_up(static_cast<size_t>(N) * 4, 256);
  p.off_frows = o;
  o += round_up(static_cast<size_t>(N) * 4, 256);
  p.fused_bytes = o;
  return p;
}

static int flce_checks(const void* H, const void* W, int dt, int64_t N, int64_t D, int64_t V,
                       const int64_t* labels, int reduction) {
  if (!valid_dtype(dt)) return FLCE_EDTYPE;
  if (!valid_reduction(reduction)) return FLCE_EINVAL;
  if (N < 0 || D < 8 || V < 1 || V >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      D >= (int64_t(1) << 31))
    return FLCE_ESHAPE;
  // N == 0 (an empty batch) is valid; H and labels may then be null
  if (W == nullptr || (N > 0 && (H == nullptr || labels == nullptr))) return FLCE_EINVAL;
  if (!aligned(H, 16) || !aligned(W, 16) || (D * static_cast<int64_t>(dtype_size(dt))) % 16 != 0)
    return FLCE_EALIGN;
  if (!aligned(labels, 8)) return FLCE_EALIGN;
  return FLCE_OK;
}

}  // namespace flce

using namespace flce;

extern "C" int64_t flce_default_chunk(int dt, int64_t N, int64_t D, int64_t V) {
  if (!valid_dtype(dt) || N < 1 || V < 1 || D < 1) return 0;
  return default_chunk(dt, N, D, V);
}

extern "C" size_t flce_workspace_bytes(int dt, int64_t N, int64_t D, int64_t V, int64_t chunk) {
  if (!valid_dtype(dt) || N < 1 || V < 1) return 0;
  return plan(dt, N, D, V, chunk, /*bwd_split=*/true).total;
}

// Forward contraction of one (shard of the) vocabulary: per (row, 256-column
// tile) partials and the label logit into the workspace.  v0 is the vocabulary
// id of W's row 0 (0 unsharded).
static int fwd_gemm(const void* H, const void* W, const void* bias, int dt, int64_t N, int64_t D,
                    int64_t V, int64_t v0, const int64_t* labels, int64_t ignore_index,
                    const FlcePlan& p, char* w, int32_t* status, cudaStream_t s) {
  float* part_m = reinterpret_cast<float*>(w + p.off_part_m);
  float* part_s = reinterpret_cast<float*>(w + p.off_part_s);
  float* zlab = reinterpret_cast<float*>(w + p.off_zlab);
  const Operand a{H, N, D, D, false};
  const Operand b{W, V, D, D, false};
  const int group = group_for(D, dt, static_cast<int>((N + kBM - 1) / kBM));
  if (dt == FLCE_BF16) {
    using E = EpiLse<__nv_bfloat16>;
    E::Params ep{bias, labels, ignore_index, static_cast<int>(N), static_cast<int>(V),
                 p.part_ld, part_m, part_s, zlab, v0};
    ep.status = status;
    return launch_gemm<__nv_bfloat16, kBNFwd, false, false, E>(kRoleFwd, a, b, nullptr, (int)N,
                                                               (int)V, (int)D, group, ep, status,
                                                               s);
  }
  using E = EpiLse<float>;
  E::Params ep{bias, labels, ignore_index, static_cast<int>(N), static_cast<int>(V), p.part_ld,
               part_m, part_s, zlab, v0};
  ep.status = status;
  return launch_gemm<float, kBNFwd, false, false, E>(kRoleFwd, a, b, nullptr, (int)N, (int)V,
                                                     (int)D, group, ep, status, s);
}

extern "C" int flce_fwd(const void* H, const void* W, const void* bias, int dt, int64_t N,
                        int64_t D, int64_t V, const int64_t* labels, int64_t ignore_index,
                        int reduction, int64_t num_label_tokens, float* loss, int64_t* n_valid,
                        float* lse, float* loss_rows, float* label_logit, void* ws,
                        size_t ws_bytes, int32_t* status, flce_stream_t stream) {
  int rc = flce_checks(H, W, dt, N, D, V, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (loss == nullptr || n_valid == nullptr || status == nullptr || (N > 0 && lse == nullptr))
    return FLCE_EINVAL;
  if (bias != nullptr && !aligned(bias, dtype_size(dt))) return FLCE_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0)  // loss 0, n_valid 0
    return launch_finalize(nullptr, labels, 0, V, ignore_index, reduction, num_label_tokens,
                           loss, n_valid, s);
  const FlcePlan p = plan(dt, N, D, V, 0);
  if (ws == nullptr || ws_bytes < p.fwd_bytes) return FLCE_EWORKSPACE;
  if (!aligned(ws, 256)) return FLCE_EALIGN;
  rc = bind_context();
  if (rc != FLCE_OK) return rc;
  char* w = static_cast<char*>(ws);
  float* rows = loss_rows != nullptr ? loss_rows : reinterpret_cast<float*>(w + p.off_rows);
  rc = fwd_gemm(H, W, bias, dt, N, D, V, 0, labels, ignore_index, p, w, status, s);
  if (rc != FLCE_OK) return rc;
  lse_combine_kernel<<<static_cast<unsigned>((N + kCombineRows - 1) / kCombineRows),
                       combine_threads(p.nparts), 0, s>>>(
      reinterpret_cast<float*>(w + p.off_part_m), reinterpret_cast<float*>(w + p.off_part_s),
      p.nparts, p.part_ld, reinterpret_cast<float*>(w + p.off_zlab), labels, N, V, ignore_index,
      lse, rows, label_logit, status);
  rc = launch_status("lse_combine_kernel launch");
  if (rc != FLCE_OK) return rc;
  return launch_finalize(rows, labels, N, V, ignore_index, reduction, num_label_tokens, loss,
                         n_valid, s);
}

extern "C" int flce_fwd_shard(const void* H, const void* W_shard, const void* bias_shard, int dt,
                              int64_t N, int64_t D, int64_t V_shard, int64_t vocab_offset,
                              int64_t V_total, const int64_t* labels, int64_t ignore_index,
                              float* m_local, float* s_local, float* zy_local, void* ws,
                              size_t ws_bytes, int32_t* status, flce_stream_t stream) {
  int rc = flce_checks(H, W_shard, dt, N, D, V_shard, labels, FLCE_SUM);
  if (rc != FLCE_OK) return rc;
  if (vocab_offset < 0 || V_total < vocab_offset + V_shard || V_total >= (int64_t(1) << 31))
    return FLCE_ESHAPE;
  if (status == nullptr ||
      (N > 0 && (m_local == nullptr || s_local == nullptr || zy_local == nullptr)))
    return FLCE_EINVAL;
  if (bias_shard != nullptr && !aligned(bias_shard, dtype_size(dt))) return FLCE_EALIGN;
  if (N == 0) return FLCE_OK;  // no rows, no partials
  const FlcePlan p = plan(dt, N, D, V_shard, 0);
  if (ws == nullptr || ws_bytes < p.fwd_bytes) return FLCE_EWORKSPACE;
  if (!aligned(ws, 256)) return FLCE_EALIGN;
  rc = bind_context();
  if (rc != FLCE_OK) return rc;
  char* w = static_cast<char*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = fwd_gemm(H, W_shard, bias_shard, dt, N, D, V_shard, vocab_offset, labels, ignore_index, p,
                w, status, s);
  if (rc != FLCE_OK) return rc;
  shard_combine_kernel<<<static_cast<unsigned>((N + kCombineRows - 1) / kCombineRows),
                         combine_threads(p.nparts), 0, s>>>(
      reinterpret_cast<float*>(w + p.off_part_m), reinterpret_cast<float*>(w + p.off_part_s),
      p.nparts, p.part_ld, reinterpret_cast<float*>(w + p.off_zlab), labels, N, V_shard,
      vocab_offset, ignore_index, m_local, s_local, zy_local);
  return launch_status("shard_combine_kernel launch");
}

extern "C" int flce_shard_rescale(const float* m_local, const float* s_local,
                                  const float* m_global, int64_t N, float* s_scaled,
                                  flce_stream_t stream) {
  if (N < 0) return FLCE_ESHAPE;
  if (N == 0) return FLCE_OK;
  if (m_local == nullptr || s_local == nullptr || m_global == nullptr || s_scaled == nullptr)
    return FLCE_EINVAL;
  shard_rescale_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(m_local, s_local, m_global, N,
                                                                   s_scaled);
  return launch_status("shard_rescale_kernel launch");
}

extern "C" int flce_shard_finish(const float* m_global, const float* s_global,
                                 const float* zy_global, const int64_t* labels, int64_t N,
                                 int64_t V_total, int64_t ignore_index, int reduction,
                                 int64_t num_label_tokens, float* lse, float* loss_rows,
                                 float* loss, int64_t* n_valid, void* ws, size_t ws_bytes,
                                 int32_t* status, flce_stream_t stream) {
  if (!valid_reduction(reduction)) return FLCE_EINVAL;
  if (N < 0 || V_total < 1 || V_total >= (int64_t(1) << 31)) return FLCE_ESHAPE;
  if (loss == nullptr || n_valid == nullptr || status == nullptr ||
      (N > 0 && (m_global == nullptr || s_global == nullptr || zy_global == nullptr ||
                 labels == nullptr || lse == nullptr)))
    return FLCE_EINVAL;
  if (N == 0)  // loss 0, n_valid 0
    return launch_finalize(nullptr, labels, 0, V_total, ignore_index, reduction,
                           num_label_tokens, loss, n_valid, reinterpret_cast<cudaStream_t>(stream));
  float* rows = loss_rows;
  if (rows == nullptr) {
    if (ws == nullptr || ws_bytes < round_up(static_cast<size_t>(N) * 4, 256))
      return FLCE_EWORKSPACE;
    rows = static_cast<float*>(ws);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  shard_finish_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0, s>>>(
      m_global, s_global, zy_global, labels, N, V_total, ignore_index, lse, rows, status);
  int rc = launch_status("shard_finish_kernel launch");
  if (rc != FLCE_OK) return rc;
  return launch_finalize(rows, labels, N, V_total, ignore_index, reduction, num_label_tokens,
                         loss, n_valid, s);
}

// The dZ contraction of the backward (step 1).  At a short K (K = D <= 1024)
// the dZ epilogue, which forms and stores a bf16 tile, is as long as the
// tile's main loop; eight epilogue warps (two per TMEM lane quarter) halve
// it.  At a long K four warps keep up (eight, for every contraction, made the
// Llama-3 8B head's step 1.7% slower).
template <typename T>
static bool dz_wide(int64_t K) {
  return sizeof(T) == 2 && K <= 1024 && (g_pair_mask.load() & kWideDz) != 0;
}

template <typename T>
static int launch_dz_gemm(const Operand& a, const Operand& b, const OutDesc& o, int M, int N,
                          int K, int group_m, const typename EpiDlogits<T>::Params& ep,
                          int32_t* status, cudaStream_t s, bool wide) {
  using E = EpiDlogits<T>;
  if constexpr (sizeof(T) == 2) {
    if (wide)
      return launch_gemm<T, kBNFwd, false, false, E, 8>(kRoleDz, a, b, &o, M, N, K, group_m, ep,
                                                        status, s);
  }
  return launch_gemm<T, kBNFwd, false, false, E>(kRoleDz, a, b, &o, M, N, K, group_m, ep,
                                                 status, s);
}

// Steps 2-4 of a backward chunk, shared by flce_bwd and flce_fwd_bwd: bias
// column sums, grad_H of the chunk, grad_W accumulation, from the chunk's dZ.
//
// grad_H_f32: grad_H_chunk is fp32 whatever the input dtype (the partial of a
// vocabulary shard, summed over the ranks before one rounding).
//
// grad_H_acc_beta >= 0 (vocabulary slices, bf16): grad_H_chunk is an fp32
// accumulator that this slice's term is stored into (0) or reduce-added to (1).
//
// dz_colsum_parts > 0: the dZ epilogue has already written that many rows of
// partial column sums (row stride p.ldV) into the column-sum buffer.
template <typename T>
static int bwd_tail(const void* W, const T* Hc, int64_t D, int64_t V, int C, bool first_chunk,
                    const FlcePlan& p, char* w, void* grad_H_chunk, float* grad_W,
                    int accumulate_grad_W, float* grad_bias, int32_t* status, cudaStream_t s,
                    bool grad_H_f32 = false, int grad_H_acc_beta = -1,
                    int dz_colsum_parts = 0) {
  const int dt = sizeof(T) == 2 ? FLCE_BF16 : FLCE_F32;
  const int dt_h = grad_H_f32 ? FLCE_F32 : dt;
  constexpr bool kTf32 = sizeof(T) == 4;
  T* dz = reinterpret_cast<T*>(w + p.off_dz);
  float* colsum = reinterpret_cast<float*>(w + p.off_colsum);
  float* Wt = reinterpret_cast<float*>(w + p.off_Wt);    // [D, ldVt]  (fp32 only)
  float* dzT = reinterpret_cast<float*>(w + p.off_dzT);  // [V, ldCt]  (fp32 only)
  float* HT = reinterpret_cast<float*>(w + p.off_HT);    // [D, ldCt]  (fp32 only)
  int rc = FLCE_OK;
  // 2. bias gradient: the column sums of dZ, from the dZ epilogue's partial
  // sums or from partial sums over row slices of the stored dZ; the partial
  // rows are added up by the epilogue warps of the next contraction before
  // their first tile (bias_pre), or by a kernel of their own when no
  // contraction follows
  EpiPre bias_pre;
  if (grad_bias != nullptr) {
    int nparts = dz_colsum_parts;
    int64_t ld = p.ldV;
    if (nparts == 0) {
      constexpr int kEpv = Elem<T>::kPerVec;
      dim3 g1(static_cast<unsigned>(((V + kEpv - 1) / kEpv + 255) / 256), kColSplits);
      colsum_partial_kernel<T><<<g1, 256, 0, s>>>(dz, C, p.ldV, (int)V, colsum);
      nparts = kColSplits;
      ld = V;
    }
    if (grad_H_chunk != nullptr || grad_W != nullptr) {
      bias_pre.kind = 1;
      bias_pre.part = colsum;
      bias_pre.nparts = nparts;
      bias_pre.ld = ld;
      bias_pre.n = V;
      bias_pre.out = grad_bias;
      bias_pre.beta = first_chunk ? 0 : 1;
    } else {
      colsum_final_kernel<<<static_cast<unsigned>((V + 31) / 32), 32 * kColFinalWarps, 0, s>>>(
          colsum, nparts, ld, (int)V, grad_bias, first_chunk ? 0 : 1);
    }
    rc = launch_status("colsum kernels launch");
    if (rc != FLCE_OK) return rc;
  }
  // the closing work that grad_W's epilogue warps take on (see bias_pre)
  EpiPre w_pre;
  // 3. grad_H[chunk] = dZ W
  const int S =
      grad_H_chunk != nullptr && grad_H_acc_beta < 0 ? grad_h_splits(C, D, V, dt) : 1;
  if (grad_H_chunk != nullptr && grad_H_acc_beta >= 0) {
    if constexpr (sizeof(T) == 2) {
      using E = EpiStore<float, true>;
      typename E::Params ep{C, static_cast<int>(D), grad_H_acc_beta};
      const Operand a{dz, C, V, p.ldV, false};
      const Operand b{W, D, V, D, true};
      const OutDesc o{grad_H_chunk, FLCE_F32, C, D, D};
      rc = launch_gemm<T, 256, false, true, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                               status, s, 1, bias_pre);
      if (rc != FLCE_OK) return rc;
    } else {
      return FLCE_ENOSUP;
    }
  } else if (grad_H_chunk != nullptr && S > 1) {
    // few output tiles: split K (= V), fp32 partials, fixed-order reduction
    const int64_t rows = static_cast<int64_t>((C + kBM - 1) / kBM) * kBM;
    float* hpart = reinterpret_cast<float*>(w + p.off_hpart);
    using E = EpiStore<float, false>;
    typename E::Params ep{static_cast<int>(S * rows), static_cast<int>(D), 0};
    const Operand a{dz, C, V, p.ldV, false};
    const OutDesc o{hpart, FLCE_F32, S * rows, D, D};
    if (kTf32) {
      const Operand b{reinterpret_cast<float*>(w + p.off_Wt), D, V, p.ldVt, false};
      rc = launch_gemm<T, 256, false, false, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                                status, s, S, bias_pre);
    } else {
      const Operand b{W, D, V, D, true};
      rc = launch_gemm<T, 256, false, true, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                               status, s, S, bias_pre);
    }
    if (rc != FLCE_OK) return rc;
    const int64_t n = static_cast<int64_t>(C) * D / 4;
    if (grad_W != nullptr) {  // closed by grad_W's epilogue warps
      w_pre.kind = 2;
      w_pre.part = hpart;
      w_pre.nparts = S;
      w_pre.ld = rows * D;
      w_pre.n = n;
      w_pre.out = grad_H_chunk;
      w_pre.out_bf16 = !grad_H_f32 && sizeof(T) == 2 ? 1 : 0;
    } else {
      const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, sm_count() * 8));
      if (grad_H_f32)
        splitk_reduce_kernel<float><<<grid, 256, 0, s>>>(hpart, S, rows * D, C, (int)D,
                                                         static_cast<float*>(grad_H_chunk));
      else
        splitk_reduce_kernel<T><<<grid, 256, 0, s>>>(hpart, S, rows * D, C, (int)D,
                                                     static_cast<T*>(grad_H_chunk));
      rc = launch_status("splitk_reduce_kernel launch");
      if (rc != FLCE_OK) return rc;
    }
  } else if (grad_H_chunk != nullptr && grad_H_f32 && !kTf32) {
    // bf16 operands, fp32 output: the split-K partial's epilogue with one split
    using E = EpiStore<float, false>;
    typename E::Params ep{C, static_cast<int>(D), 0};
    const Operand a{dz, C, V, p.ldV, false};
    const OutDesc o{grad_H_chunk, FLCE_F32, C, D, D};
    const Operand b{W, D, V, D, true};
    rc = launch_gemm<T, 256, false, true, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                             status, s, 1, bias_pre);
    if (rc != FLCE_OK) return rc;
  } else if (grad_H_chunk != nullptr) {
    using E = EpiStore<T, false>;
    typename E::Params ep{C, static_cast<int>(D), 0};
    const Operand a{dz, C, V, p.ldV, false};
    const OutDesc o{grad_H_chunk, dt_h, C, D, D};
    if (kTf32) {
      const Operand b{Wt, D, V, p.ldVt, false};
      rc = launch_gemm<T, 256, false, false, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                                status, s, 1, bias_pre);
    } else {
      const Operand b{W, D, V, D, true};
      rc = launch_gemm<T, 256, false, true, E>(kRoleGradH, a, b, &o, C, (int)D, (int)V, 8, ep,
                                               status, s, 1, bias_pre);
    }
    if (rc != FLCE_OK) return rc;
  }
  // 4. grad_W (+)= dZ^T H[chunk]
  if (grad_H_chunk == nullptr) w_pre = bias_pre;  // no grad_H launch took the bias sums
  if (grad_W != nullptr) {
    using E = EpiStore<float, true>;
    typename E::Params ep{static_cast<int>(V), static_cast<int>(D),
                          (!first_chunk || accumulate_grad_W) ? 1 : 0};
    const OutDesc o{grad_W, FLCE_F32, V, D, D};
    if (kTf32) {
      transpose32(reinterpret_cast<const float*>(dz), C, (int)V, p.ldV, dzT, p.ldCt, s);
      transpose32(reinterpret_cast<const float*>(Hc), C, (int)D, D, HT, p.ldCt, s);
      rc = launch_status("transpose32(dZ, H) launch");
      if (rc != FLCE_OK) return rc;
      const Operand a{dzT, V, C, p.ldCt, false};
      const Operand b{HT, D, C, p.ldCt, false};
      rc = launch_gemm<T, 256, false, false, E>(kRoleGradW, a, b, &o, (int)V, (int)D, C, 8, ep,
                                                status, s, 1, w_pre);
    } else {
      const Operand a{dz, V, C, p.ldV, true};
      const Operand b{Hc, D, C, D, true};
      rc = launch_gemm<T, 256, true, true, E>(kRoleGradW, a, b, &o, (int)V, (int)D, C, 8, ep,
                                              status, s, 1, w_pre);
    }
    if (rc != FLCE_OK) return rc;
  }
  return rc;
}

template <typename T>
static int transpose_W_if_needed(const void* W, int64_t D, int64_t V, const FlcePlan& p, char* w,
                                 void* grad_H, cudaStream_t s) {
  if (sizeof(T) != 4 || grad_H == nullptr) return FLCE_OK;
  transpose32(static_cast<const float*>(W), (int)V, (int)D, D,
              reinterpret_cast<float*>(w + p.off_Wt), p.ldVt, s);
  return launch_status("transpose32(W) launch");
}

template <typename T>
static int flce_bwd_impl(const void* H, const void* W, const void* bias, int64_t N, int64_t D,
                         int64_t V, int64_t v0, int64_t V_total, const int64_t* labels,
                         int64_t ignore_index, int reduction,
                         int64_t num_label_tokens, const float* lse, const int64_t* n_valid,
                         const float* grad_loss, const FlcePlan& p, void* grad_H,
                         float* grad_W, int accumulate_grad_W, float* grad_bias, char* w,
                         int32_t* status, cudaStream_t s, bool grad_H_f32 = false) {
  const int dt = sizeof(T) == 2 ? FLCE_BF16 : FLCE_F32;
  T* dz = reinterpret_cast<T*>(w + p.off_dz);
  const T* Ht = static_cast<const T*>(H);
  const size_t h_es = grad_H_f32 ? sizeof(float) : sizeof(T);
  int rc = FLCE_OK;
  if constexpr (sizeof(T) == 2) {
    if (p.vchunk > 0) {
      // Vocabulary slices: per slice of columns [c0, c0 + Vc), dZ of all rows,
      // the slice's bias columns, its rows of grad_W (written once), and its
      // term of grad_H accumulated in fp32; then grad_H rounded once.
      FlcePlan pv = p;
      pv.ldV = p.ldVc;
      float* hacc = grad_H_f32 ? static_cast<float*>(grad_H)
                               : reinterpret_cast<float*>(w + p.off_hacc);
      const T* bias_t = static_cast<const T*>(bias);
      const int nMt = static_cast<int>((N + kBM - 1) / kBM);
      int k = 0;
      for (int64_t c0 = 0; c0 < V; c0 += p.vchunk, ++k) {
        const int Vc = static_cast<int>(std::min<int64_t>(p.vchunk, V - c0));
        const T* Wc = static_cast<const T*>(W) + c0 * D;
        using E = EpiDlogits<T>;
        typename E::Params ep{bias_t != nullptr ? bias_t + c0 : nullptr, labels, ignore_index,
                              lse, reduction, num_label_tokens, n_valid, grad_loss,
                              static_cast<int>(N), Vc, v0 + c0, V_total};
        const bool wide = dz_wide<T>(D);
        const int parts = wide && grad_bias != nullptr
                              ? static_cast<int>(dz_colsum_rows(dt, D, N)) : 0;
        if (parts > 0) {
          ep.colsum = reinterpret_cast<float*>(w + pv.off_colsum);
          ep.colsum_ld = pv.ldV;
        }
        const Operand a{Ht, N, D, D, false};
        const Operand b{Wc, Vc, D, D, false};
        const OutDesc o{dz, dt, N, Vc, p.ldVc};
        rc = launch_dz_gemm<T>(a, b, o, static_cast<int>(N), Vc, (int)D, group_for(D, dt, nMt),
                               ep, status, s, wide);
        if (rc != FLCE_OK) return rc;
        rc = bwd_tail<T>(Wc, Ht, D, Vc, static_cast<int>(N), /*first_chunk=*/true, pv, w,
                         grad_H != nullptr ? hacc : nullptr,
                         grad_W != nullptr ? grad_W + c0 * D : nullptr, accumulate_grad_W,
                         grad_bias != nullptr ? grad_bias + c0 : nullptr, status, s, false,
                         /*grad_H_acc_beta=*/k > 0 ? 1 : 0, parts);
        if (rc != FLCE_OK) return rc;
      }
      if (grad_H != nullptr && !grad_H_f32) {
        const int64_t n = N * D / 4;
        const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, sm_count() * 8));
        splitk_reduce_kernel<T><<<grid, 256, 0, s>>>(hacc, 1, N * D, static_cast<int>(N), (int)D,
                                                     static_cast<T*>(grad_H));
        rc = launch_status("splitk_reduce_kernel launch");
      }
      return rc;
    }
  }
  rc = transpose_W_if_needed<T>(W, D, V, p, w, grad_H, s);
  if (rc != FLCE_OK) return rc;
  for (int64_t r0 = 0; r0 < N; r0 += p.chunk) {
    const int C = static_cast<int>(std::min<int64_t>(p.chunk, N - r0));
    const int nMt = (C + kBM - 1) / kBM;
    // 1. recompute logits, form dZ
    using E = EpiDlogits<T>;
    typename E::Params ep{bias, labels + r0, ignore_index, lse + r0, reduction,
                          num_label_tokens, n_valid, grad_loss, C, static_cast<int>(V), v0,
                          V_total};
    // the eight-warp epilogue also forms the bias gradient's column sums
    const bool wide = dz_wide<T>(D);
    const int parts = wide && grad_bias != nullptr ? static_cast<int>(dz_colsum_rows(dt, D, C)) : 0;
    if (parts > 0) {
      ep.colsum = reinterpret_cast<float*>(w + p.off_colsum);
      ep.colsum_ld = p.ldV;
    }
    const Operand a{Ht + r0 * D, C, D, D, false};
    const Operand b{W, V, D, D, false};
    const OutDesc o{dz, dt, C, V, p.ldV};
    rc = launch_dz_gemm<T>(a, b, o, C, (int)V, (int)D, group_for(D, dt, nMt), ep, status, s,
                           wide);
    if (rc != FLCE_OK) return rc;
    rc = bwd_tail<T>(W, Ht + r0 * D, D, V, C, r0 == 0, p, w,
                     grad_H != nullptr ? static_cast<char*>(grad_H) + r0 * D * h_es : nullptr,
                     grad_W, accumulate_grad_W, grad_bias, status, s, grad_H_f32, -1, parts);
    if (rc != FLCE_OK) return rc;
  }
  return rc;
}

// Fused forward + backward: per chunk, the forward GEMM also stores the
// chunk's logits (as offsets u from each tile's maximum), the chunk's lse is
// combined, dZ is formed in place from u, then steps 2-4 as in flce_bwd.
template <typename T>
static int flce_fused_impl(const void* H, const void* W, const void* bias, int64_t N, int64_t D,
                           int64_t V, const int64_t* labels, int64_t ignore_index,
                           int reduction, int64_t num_label_tokens, const float* grad_loss,
                           const FlcePlan& p, float* loss, int64_t* n_valid, float* lse,
                           float* loss_rows, void* grad_H, float* grad_W, int accumulate_grad_W,
                           float* grad_bias, char* w, int32_t* status, cudaStream_t s) {
  const int dt = sizeof(T) == 2 ? FLCE_BF16 : FLCE_F32;
  T* dz = reinterpret_cast<T*>(w + p.off_dz);
  float* part_m = reinterpret_cast<float*>(w + p.off_fpart_m);
  float* part_s = reinterpret_cast<float*>(w + p.off_fpart_s);
  float* zlab = reinterpret_cast<float*>(w + p.off_fzlab);
  float* rows = loss_rows != nullptr ? loss_rows : reinterpret_cast<float*>(w + p.off_frows);
  const T* Ht = static_cast<const T*>(H);
  count_valid_kernel<<<1, 1024, 0, s>>>(labels, N, V, ignore_index, n_valid);
  int rc = launch_status("count_valid_kernel launch");
  if (rc != FLCE_OK) return rc;
  rc = transpose_W_if_needed<T>(W, D, V, p, w, grad_H, s);
  if (rc != FLCE_OK) return rc;
  for (int64_t r0 = 0; r0 < N; r0 += p.chunk) {
    const int C = static_cast<int>(std::min<int64_t>(p.chunk, N - r0));
    const int nMt = (C + kBM - 1) / kBM;
    // 1. logits of the chunk: lse partials and u into the chunk buffer
    {
      using E = EpiLseStore<T>;
      typename E::Params ep{bias, labels + r0, ignore_index, C, static_cast<int>(V),
                            p.fpart_ld, part_m, part_s, zlab + r0};
      ep.status = status;
      const Operand a{Ht + r0 * D, C, D, D, false};
      const Operand b{W, V, D, D, false};
      const OutDesc o{dz, dt, C, V, p.ldV};
      rc = launch_gemm<T, kBNFwd, false, false, E>(kRoleFwd, a, b, &o, C, (int)V, (int)D,
                                                   group_for(D, dt, nMt), ep, status, s);
      if (rc != FLCE_OK) return rc;
    }
    // 2. lse and per-row loss of the chunk
    lse_combine_kernel<<<static_cast<unsigned>((C + kCombineRows - 1) / kCombineRows),
                         combine_threads(p.nparts), 0, s>>>(
        part_m, part_s, p.nparts, p.fpart_ld, zlab + r0, labels + r0, C, V, ignore_index,
        lse + r0, rows + r0, nullptr, status);
    // 3. dZ in place
    {
      const int grid = std::min(C, sm_count() * 8);
      dz_from_u_kernel<T><<<grid, 256, p.nparts * sizeof(float), s>>>(
          dz, C, (int)V, p.ldV, part_m, p.nparts, p.fpart_ld, lse + r0, labels + r0,
          ignore_index, reduction, num_label_tokens, n_valid, grad_loss);
    }
    rc = launch_status("lse_combine / dz_from_u launch");
    if (rc != FLCE_OK) return rc;
    rc = bwd_tail<T>(W, Ht + r0 * D, D, V, C, r0 == 0, p, w,
                     grad_H != nullptr ? static_cast<T*>(grad_H) + r0 * D : nullptr, grad_W,
                     accumulate_grad_W, grad_bias, status, s);
    if (rc != FLCE_OK) return rc;
  }
  return launch_finalize(rows, labels, N, V, ignore_index, reduction, num_label_tokens, loss,
                         n_valid, s);
}

static int flce_bwd_entry(const void* H, const void* W, const void* bias, int dt, int64_t N,
                          int64_t D, int64_t V, int64_t v0, int64_t V_total,
                          const int64_t* labels, int64_t ignore_index, int reduction,
                          int64_t num_label_tokens, const float* lse, const int64_t* n_valid,
                          const float* grad_loss, int64_t chunk, void* grad_H, float* grad_W,
                          int accumulate_grad_W, float* grad_bias, void* ws, size_t ws_bytes,
                          int32_t* status, flce_stream_t stream, bool grad_H_f32 = false) {
  int rc = flce_checks(H, W, dt, N, D, V, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (v0 < 0 || V_total < v0 + V || V_total >= (int64_t(1) << 31)) return FLCE_ESHAPE;
  if (n_valid == nullptr || grad_loss == nullptr || status == nullptr ||
      (N > 0 && lse == nullptr))
    return FLCE_EINVAL;
  if (accumulate_grad_W != 0 && accumulate_grad_W != 1) return FLCE_EINVAL;
  if (chunk > 0 && chunk % kBM != 0 && chunk < N) return FLCE_ESHAPE;
  if (chunk < 0 && dt != FLCE_BF16) return FLCE_ENOSUP;  // vocabulary slices: bf16 only
  if (chunk < 0 && (-chunk) % 256 != 0) return FLCE_ESHAPE;
  if (bias != nullptr && !aligned(bias, dtype_size(dt))) return FLCE_EALIGN;
  if (grad_H != nullptr && !aligned(grad_H, 16)) return FLCE_EALIGN;
  if (grad_W != nullptr && !aligned(grad_W, 16)) return FLCE_EALIGN;
  if (grad_bias != nullptr && !aligned(grad_bias, 4)) return FLCE_EALIGN;
  if (N == 0)
    return empty_bwd(D, V, grad_W, accumulate_grad_W, grad_bias,
                     reinterpret_cast<cudaStream_t>(stream));
  const FlcePlan p = plan(dt, N, D, V, chunk, /*bwd_split=*/true);
  if (ws == nullptr || ws_bytes < p.bwd_bytes) return FLCE_EWORKSPACE;
  if (!aligned(ws, 256)) return FLCE_EALIGN;
  if (grad_H == nullptr && grad_W == nullptr && grad_bias == nullptr) return FLCE_OK;
  rc = bind_context();
  if (rc != FLCE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  if (dt == FLCE_BF16)
    return flce_bwd_impl<__nv_bfloat16>(H, W, bias, N, D, V, v0, V_total, labels, ignore_index,
                                        reduction, num_label_tokens, lse, n_valid, grad_loss, p,
                                        grad_H, grad_W, accumulate_grad_W, grad_bias, w, status,
                                        s, grad_H_f32);
  return flce_bwd_impl<float>(H, W, bias, N, D, V, v0, V_total, labels, ignore_index, reduction,
                              num_label_tokens, lse, n_valid, grad_loss, p, grad_H, grad_W,
                              accumulate_grad_W, grad_bias, w, status, s);
}

extern "C" int flce_bwd(const void* H, const void* W, const void* bias, int dt, int64_t N,
                        int64_t D, int64_t V, const int64_t* labels, int64_t ignore_index,
                        int reduction, int64_t num_label_tokens, const float* lse,
                        const int64_t* n_valid, const float* grad_loss, int64_t chunk,
                        void* grad_H, float* grad_W, int accumulate_grad_W, float* grad_bias,
                        void* ws, size_t ws_bytes, int32_t* status, flce_stream_t stream) {
  return flce_bwd_entry(H, W, bias, dt, N, D, V, 0, V, labels, ignore_index, reduction,
                        num_label_tokens, lse, n_valid, grad_loss, chunk, grad_H, grad_W,
                        accumulate_grad_W, grad_bias, ws, ws_bytes, status, stream);
}

extern "C" int flce_bwd_shard(const void* H, const void* W_shard, const void* bias_shard,
                              int dt, int64_t N, int64_t D, int64_t V_shard,
                              int64_t vocab_offset, int64_t V_total, const int64_t* labels,
                              int64_t ignore_index, int reduction, int64_t num_label_tokens,
                              const float* lse, const int64_t* n_valid, const float* grad_loss,
                              int64_t chunk, void* grad_H_partial, float* grad_W_shard,
                              int accumulate_grad_W, float* grad_bias_shard, void* ws,
                              size_t ws_bytes, int32_t* status, flce_stream_t stream) {
  return flce_bwd_entry(H, W_shard, bias_shard, dt, N, D, V_shard, vocab_offset, V_total, labels,
                        ignore_index, reduction, num_label_tokens, lse, n_valid, grad_loss,
                        chunk, grad_H_partial, grad_W_shard, accumulate_grad_W, grad_bias_shard,
                        ws, ws_bytes, status, stream, /*grad_H_f32=*/true);
}

extern "C" size_t flce_fwd_bwd_workspace_bytes(int dt, int64_t N, int64_t D, int64_t V,
                                               int64_t chunk) {
  if (!valid_dtype(dt) || N < 1 || V < 1) return 0;
  return plan(dt, N, D, V, chunk > 0 ? chunk : 0).fused_bytes;
}

extern "C" int flce_fwd_bwd(const void* H, const void* W, const void* bias, int dt, int64_t N,
                            int64_t D, int64_t V, const int64_t* labels, int64_t ignore_index,
                            int reduction, int64_t num_label_tokens, const float* grad_loss,
                            int64_t chunk, float* loss, int64_t* n_valid, float* lse,
                            float* loss_rows, void* grad_H, float* grad_W, int accumulate_grad_W,
                            float* grad_bias, void* ws, size_t ws_bytes, int32_t* status,
                            flce_stream_t stream) {
  int rc = flce_checks(H, W, dt, N, D, V, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (loss == nullptr || n_valid == nullptr || status == nullptr || (N > 0 && lse == nullptr))
    return FLCE_EINVAL;
  if (accumulate_grad_W != 0 && accumulate_grad_W != 1) return FLCE_EINVAL;
  if (chunk > 0 && chunk % kBM != 0 && chunk < N) return FLCE_ESHAPE;
  if (bias != nullptr && !aligned(bias, dtype_size(dt))) return FLCE_EALIGN;
  if (grad_H != nullptr && !aligned(grad_H, 16)) return FLCE_EALIGN;
  if (grad_W != nullptr && !aligned(grad_W, 16)) return FLCE_EALIGN;
  if (grad_bias != nullptr && !aligned(grad_bias, 4)) return FLCE_EALIGN;
  if (N == 0) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = launch_finalize(nullptr, labels, 0, V, ignore_index, reduction, num_label_tokens, loss,
                         n_valid, s);
    if (rc != FLCE_OK) return rc;
    return empty_bwd(D, V, grad_W, accumulate_grad_W, grad_bias, s);
  }
  const FlcePlan p = plan(dt, N, D, V, chunk > 0 ? chunk : 0);
  if (p.nparts > kMaxTilesPerRow) return FLCE_ESHAPE;
  if (ws == nullptr || ws_bytes < p.fused_bytes) return FLCE_EWORKSPACE;
  if (!aligned(ws, 256)) return FLCE_EALIGN;
  rc = bind_context();
  if (rc != FLCE_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  if (dt == FLCE_BF16)
    return flce_fused_impl<__nv_bfloat16>(H, W, bias, N, D, V, labels, ignore_index, reduction,
                                          num_label_tokens, grad_loss, p, loss, n_valid, lse,
                                          loss_rows, grad_H, grad_W, accumulate_grad_W,
                                          grad_bias, w, status, s);
  return flce_fused_impl<float>(H, W, bias, N, D, V, labels, ignore_index, reduction,
                                num_label_tokens, grad_loss, p, loss, n_valid, lse, loss_rows,
                                grad_H, grad_W, accumulate_grad_W, grad_bias, w, status, s);
}

extern "C" int flce_count_valid(const int64_t* labels, int64_t N, int64_t V, int64_t ignore_index,
                                int64_t* n_valid, flce_stream_t stream) {
  if (N < 0 || V < 1) return FLCE_ESHAPE;
  if (n_valid == nullptr || (N > 0 && labels == nullptr)) return FLCE_EINVAL;
  if (!aligned(labels, 8) || !aligned(n_valid, 8)) return FLCE_EALIGN;
  count_valid_kernel<<<1, 1024, 0, reinterpret_cast<cudaStream_t>(stream)>>>(labels, N, V,
                                                                          ignore_index, n_valid);
  return launch_status("count_valid_kernel launch");
}

extern "C" int flce_grad_scale(void* x, int dt, int64_t n, const float* g, flce_stream_t stream) {
  if (!valid_dtype(dt)) return FLCE_EDTYPE;
  if (n < 0) return FLCE_ESHAPE;
  if (n == 0) return FLCE_OK;
  if (x == nullptr || g == nullptr) return FLCE_EINVAL;
  if (!aligned(x, dtype_size(dt))) return FLCE_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, sm_count() * 8));
  if (dt == FLCE_BF16)
    scale_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<__nv_bfloat16*>(x), n, g);
  else
    scale_kernel<float><<<grid, 256, 0, s>>>(static_cast<float*>(x), n, g);
  return launch_status("scale_kernel launch");
}

// ------------------------------------------------------ raw GEMM entry point

extern "C" int flce_gemm_set_pair(int mask) { return g_pair_mask.exchange(mask & 63); }

extern "C" int flce_gemm_pair_slots(void) {
  using E = EpiStore<float, true>;
  auto kern = tc_gemm_pair_kernel<256, false, false, E>;
  using G = PairGeo<256>;
  if (bind_context() != FLCE_OK) return -1;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) !=
      cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
  return n;
}

extern "C" int flce_gemm(int dt, int a_mn_major, int b_mn_major, int64_t M, int64_t N, int64_t K,
                         const void* A, int64_t lda, const void* B, int64_t ldb, float* C,
                         int64_t ldc, int accumulate, int32_t* status, flce_stream_t stream) {
  if (!valid_dtype(dt)) return FLCE_EDTYPE;
  if (M < 1 || N < 1 || K < 1 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
      K >= (int64_t(1) << 31))
    return FLCE_ESHAPE;
  if (A == nullptr || B == nullptr || C == nullptr || status == nullptr) return FLCE_EINVAL;
  if ((a_mn_major != 0 && a_mn_major != 1) || (b_mn_major != 0 && b_mn_major != 1) ||
      (accumulate != 0 && accumulate != 1))
    return FLCE_EINVAL;
  const int64_t es = static_cast<int64_t>(dtype_size(dt));
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16) || (lda * es) % 16 != 0 ||
      (ldb * es) % 16 != 0 || ldc % 4 != 0)
    return FLCE_EALIGN;
  if (lda < (a_mn_major ? M : K) || ldb < (b_mn_major ? N : K) || ldc < N) return FLCE_ESHAPE;
  // The tf32 tensor-core path reads K-major operands only.
  if (dt == FLCE_F32 && (a_mn_major || b_mn_major)) return FLCE_ENOSUP;
  const int brc = bind_context();
  if (brc != FLCE_OK) return brc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const Operand a{A, M, K, lda, a_mn_major != 0};
  const Operand b{B, N, K, ldb, b_mn_major != 0};
  using E = EpiStore<float, true>;
  E::Params ep{static_cast<int>(M), static_cast<int>(N), accumulate};
  const OutDesc o{C, FLCE_F32, M, N, ldc};
  const int code = (dt == FLCE_BF16 ? 0 : 4) | (a_mn_major ? 2 : 0) | (b_mn_major ? 1 : 0);
  switch (code) {
    case 0: return launch_gemm<__nv_bfloat16, 256, false, false, E>(kRoleRaw, a, b, &o, (int)M, (int)N, (int)K, 8, ep, status, s);
    case 1: return launch_gemm<__nv_bfloat16, 256, false, true, E>(kRoleRaw, a, b, &o, (int)M, (int)N, (int)K, 8, ep, status, s);
    case 2: return launch_gemm<__nv_bfloat16, 256, true, false, E>(kRoleRaw, a, b, &o, (int)M, (int)N, (int)K, 8, ep, status, s);
    case 3: return launch_gemm<__nv_bfloat16, 256, true, true, E>(kRoleRaw, a, b, &o, (int)M, (int)N, (int)K, 8, ep, status, s);
    default: return launch_gemm<float, 256, false, false, E>(kRoleRaw, a, b, &o, (int)M, (int)N, (int)K, 8, ep, status, s);
  }
}
