// Cross-entropy over given logits [N, V]: bandwidth-bound row kernels.
//
// Forward (Automodel PR #2996 "feat(loss): chunked masked CE, ...", first commit
// message): per row an fp32 log-sum-exp and the gathered label logit; the
// per-row losses are reduced to a scalar by a fixed-order fp64 sum.  The
// per-row lse (4 bytes per row) is all the backward needs besides the logits
// and labels, so the backward is one read -> write pass over the logits.
//
// Backward (same page, backward bullet and the inplace_grad commit): the
// softmax is recomputed from the logits and the saved lse, the one-hot label is
// subtracted, the result is scaled and written either into the logits storage
// (in place) or into a separate buffer.  Without a saved lse (the page's
// memory bullet: nothing but the inputs is kept) the lse is formed again in
// the backward, still with one read of the logits where the row fits a
// thread-block cluster's shared memory.  When the incoming gradient is known
// in advance, the forward and the backward run as one such pass (the
// eager-gradient scheme of Liger-Kernel issue #533, applied to given logits).
//
// Three kernel families, chosen per call:
// * ce_stream_kernel: rows stream through a cp.async.bulk shared-memory ring
//   as whole 16-byte blocks (a row that starts or ends inside a block has its
//   first and last block finished element by element): the forward; the
//   backward with a saved lse; the backward without one for rows over
//   512 KiB, read twice;
// * ce_bwd_resident_kernel: backward without a saved lse, a row held by a
//   cluster of 1-8 CTAs; in its fused mode also the forward's per-row loss
//   and lse (ce_logits_fwd_bwd: forward and backward with one read);
// * ce_bwd_rows_kernel: a backward whose gradient rows start at other offsets
//   within a 16-byte block than the logits rows (separate buffers whose
//   starts or row strides differ modulo 16 bytes): 16-byte register loads
//   with a scalar head and tail.
// All keep the online maximum and sum in the base-2 domain (one MUFU ex2 per
// element) and merge per-thread states with warp shuffles in a fixed order.
#include <math.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "host.h"

namespace flce {

// Vocabulary-shard outputs of the forward: per row the base-2 maximum and sum
// over the shard's columns and the label logit when the label lies in the shard
// (0 otherwise); labels are global ids in [0, V_total).  m_out == nullptr
// selects the ordinary (unsharded) outputs.
struct ShardOut {
  float* m_out;
  float* s_out;
  float* zy_out;
  int64_t v0;
  int64_t V_total;
  template <typename T>
  __device__ void write(int64_t row, float m, float s, int64_t y, int64_t ignore_index,
                        int64_t V_shard, const T* p, int32_t* status) const {
    m_out[row] = m;
    s_out[row] = s;
    float zy = 0.0f;
    if (y != ignore_index) {
      if (!label_ok(y, V_total))
        set_status(status, FLCE_ELABEL);
      else if (y >= v0 && y < v0 + V_shard)
        zy = Elem<T>::load(p + (y - v0));
    }
    zy_out[row] = zy;
  }
};

// ------------------------------------------------------------ row reduction

// Base-2 log-sum-exp state of one row p[0..V) over the block: every thread
// reduces a strided share (16-byte vector loads; a scalar head and tail when
// the row start is not 16-byte aligned), warps merge by shuffles, and each
// thread then merges the warp states in the same order, so all threads return
// the same state.  red_m/red_s hold THREADS/32 entries and are free again on
// return.
template <typename T, int THREADS>
__device__ Lse2 block_row_lse2(const T* p, int64_t V, float* red_m, float* red_s) {
  constexpr int EPV = Elem<T>::kPerVec;
  constexpr int UNROLL = (EPV == 8) ? 4 : 8;  // 32 elements per batch
  constexpr int NW = THREADS / 32;
  const int tid = threadIdx.x;
  Lse2 st;
  int64_t head = static_cast<int64_t>(((16u - (reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) /
                                      sizeof(T));
  if (head > V) head = V;
  for (int64_t j = tid; j < head; j += THREADS) st.add1(Elem<T>::load(p + j) * kLog2e);
  const uint4* vp = reinterpret_cast<const uint4*>(p + head);
  const int64_t nvec = (V - head) / EPV;
  int64_t v = tid;
  for (; v + (UNROLL - 1) * THREADS < nvec; v += UNROLL * THREADS) {
    uint4 u[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) u[k] = __ldcs(vp + v + k * THREADS);
    float t[UNROLL * EPV];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      float x[EPV];
      Elem<T>::unpack(u[k], x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) t[k * EPV + e] = x[e] * kLog2e;
    }
    st.addk(t);
  }
  for (; v < nvec; v += THREADS) {
    float x[EPV];
    Elem<T>::unpack(__ldcs(vp + v), x);
#pragma unroll
    for (int e = 0; e < EPV; ++e) x[e] *= kLog2e;
    st.addk(x);
  }
  for (int64_t j = head + nvec * EPV + tid; j < V; j += THREADS)
    st.add1(Elem<T>::load(p + j) * kLog2e);

#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, st.m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, st.s, o);
    st.merge(m2, s2);
  }
  if ((tid & 31) == 0) {
    red_m[tid >> 5] = st.m;
    red_s[tid >> 5] = st.s;
  }
  __syncthreads();
  Lse2 all;
  for (int w = 0; w < NW; ++w) all.merge(red_m[w], red_s[w]);
  __syncthreads();
  return all;
}

// ------------------------------------------------------------- finalize kernel

constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const float* __restrict__ loss_rows, const int64_t* __restrict__ labels, int64_t N,
    int64_t V, int64_t ignore_index, int reduction, int64_t num_label_tokens,
    float* __restrict__ loss, int64_t* __restrict__ n_valid) {
  __shared__ double sacc[kFinThreads];
  __shared__ long long scnt[kFinThreads];
  const int tid = threadIdx.x;
  double acc = 0.0;
  long long cnt = 0;
  for (int64_t i = tid; i < N; i += kFinThreads) {
    acc += static_cast<double>(loss_rows[i]);
    const int64_t y = labels[i];
    cnt += (y != ignore_index && label_ok(y, V)) ? 1 : 0;
  }
  sacc[tid] = acc;
  scnt[tid] = cnt;
  __syncthreads();
  for (int w = kFinThreads / 2; w > 0; w >>= 1) {
    if (tid < w) {
      sacc[tid] += sacc[tid + w];
      scnt[tid] += scnt[tid + w];
    }
    __syncthreads();
  }
  if (tid == 0) {
    const long long nv = scnt[0];
    int64_t div;
    if (num_label_tokens >= 0) div = num_label_tokens;
    else if (reduction == FLCE_SUM) div = 1;
    else div = nv;
    *loss = div == 0 ? 0.0f : static_cast<float>(sacc[0] / static_cast<double>(div));
    *n_valid = nv;
  }
}

int launch_finalize(const float* loss_rows, const int64_t* labels, int64_t N, int64_t V,
                    int64_t ignore_index, int reduction, int64_t num_label_tokens, float* loss,
                    int64_t* n_valid, cudaStream_t stream) {
  finalize_kernel<<<1, kFinThreads, 0, stream>>>(loss_rows, labels, N, V, ignore_index,
                                                 reduction, num_label_tokens, loss, n_valid);
  return launch_status("finalize_kernel launch");
}

// -------------------------------------------------------------- backward kernel

// The backward for a gradient buffer whose rows start at other offsets within
// their 16-byte blocks than the logits rows (the bulk-copy kernels serve every
// other case): such rows are read and written element by element (the 16-byte
// path below needs both rows at one offset).  Without a saved lse (lse ==
// nullptr) each row is reduced first (block_row_lse2), then transformed.
template <typename T, int THREADS>
__global__ void __launch_bounds__(THREADS) ce_bwd_rows_kernel(
    const T* logits, int64_t N, int64_t V, int64_t ld, const int64_t* __restrict__ labels,
    int64_t ignore_index, int reduction, int64_t num_label_tokens, const float* __restrict__ lse,
    const int64_t* n_valid, const float* grad_loss, T* grad, int64_t ldg, int64_t v0,
    int64_t V_total) {
  constexpr int EPV = Elem<T>::kPerVec;
  constexpr int UNROLL = 4;
  __shared__ float red_m[THREADS / 32], red_s[THREADS / 32];
  const float coef = grad_coef(reduction, num_label_tokens, n_valid, grad_loss);
  const int tid = threadIdx.x;

  for (int64_t row = blockIdx.x; row < N; row += gridDim.x) {
    const T* p = logits + row * ld;
    T* q = grad + row * ldg;
    const int64_t yg = labels[row];
    const bool valid = (yg != ignore_index) && label_ok(yg, V_total);
    const int64_t y = valid ? yg - v0 : -1;  // label column within this shard (or none)
    const float c = valid ? coef : 0.0f;
    float lse2;
    if (lse != nullptr) {
      lse2 = lse[row] * kLog2e;
    } else if (c != 0.0f) {  // no saved lse: a reduction pass over the row first
      const Lse2 all = block_row_lse2<T, THREADS>(p, V, red_m, red_s);
      lse2 = all.m + log2f(all.s);
    } else {
      lse2 = 0.0f;  // the row's gradient is zero
    }
    const uintptr_t pa = reinterpret_cast<uintptr_t>(p) & 15u;
    const uintptr_t qa = reinterpret_cast<uintptr_t>(q) & 15u;
    int64_t head = (pa == qa) ? static_cast<int64_t>(((16u - pa) & 15u) / sizeof(T)) : V;
    if (head > V) head = V;

    auto one = [&](int64_t j) {
      float d = 0.0f;
      if (c != 0.0f) {
        const float x = Elem<T>::load(p + j);
        d = (ex2(fmaf(x, kLog2e, -lse2)) - (j == y ? 1.0f : 0.0f)) * c;
      }
      Elem<T>::store(q + j, d);
    };
    for (int64_t j = tid; j < head; j += THREADS) one(j);
    const uint4* vp = reinterpret_cast<const uint4*>(p + head);
    uint4* vq = reinterpret_cast<uint4*>(q + head);
    const int64_t nvec = (V - head) / EPV;
    if (c == 0.0f) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int64_t v = tid; v < nvec; v += THREADS) __stcs(vq + v, z);
    } else {
      const int64_t ylocal = y - head;  // label position relative to the vector body
      int64_t v = tid;
      for (; v + (UNROLL - 1) * THREADS < nvec; v += UNROLL * THREADS) {
        uint4 u[UNROLL];
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) u[k] = __ldcs(vp + v + k * THREADS);
#pragma unroll
        for (int k = 0; k < UNROLL; ++k) {
          float x[EPV];
          Elem<T>::unpack(u[k], x);
          const int64_t j0 = (v + k * THREADS) * EPV;
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            x[e] = (ex2(fmaf(x[e], kLog2e, -lse2)) - (j0 + e == ylocal ? 1.0f : 0.0f)) * c;
          __stcs(vq + v + k * THREADS, Elem<T>::pack(x));
        }
      }
      for (; v < nvec; v += THREADS) {
        float x[EPV];
        Elem<T>::unpack(__ldcs(vp + v), x);
        const int64_t j0 = v * EPV;
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          x[e] = (ex2(fmaf(x[e], kLog2e, -lse2)) - (j0 + e == ylocal ? 1.0f : 0.0f)) * c;
        __stcs(vq + v, Elem<T>::pack(x));
      }
    }
    for (int64_t j = head + nvec * EPV + tid; j < V; j += THREADS) one(j);
  }
}

// ------------------------------------------------ bulk-copy (TMA) row streaming

// Rows are streamed through a shared-memory ring: one producer thread copies
// 32 KB segments of a row's 16-byte blocks with cp.async.bulk (a 2-stage
// mbarrier ring, so up to 64 KB per CTA is in flight without holding
// registers; 3 CTAs per SM), and 8 consumer warps reduce (forward) or
// transform and store (backward) each segment from shared memory.  The segment size, stage count and CTAs per SM were chosen by a
// sweep on GB300 (16-32 KB segments, 2-8 stages, 2-4 CTAs per SM).
#ifndef FLCE_CE_SEG_BYTES
#define FLCE_CE_SEG_BYTES 32768
#endif
#ifndef FLCE_CE_STAGES
#define FLCE_CE_STAGES 2
#endif
#ifndef FLCE_CE_CTAS_PER_SM
#define FLCE_CE_CTAS_PER_SM 3
#endif
constexpr int kSegBytes = FLCE_CE_SEG_BYTES;
constexpr int kRingStages = FLCE_CE_STAGES;
constexpr int kConsumers = 256;
constexpr int kConsumerWarps = kConsumers / 32;
constexpr int kStreamThreads = kConsumers + 32;
constexpr int kStreamSmem = kRingStages * kSegBytes + 128;
constexpr int kStreamCtasPerSm = FLCE_CE_CTAS_PER_SM;
static_assert(kSegBytes % (16 * kConsumers) == 0, "whole 16-byte vectors per consumer");

// Adds K vectors sv[first + k*STRIDE] (those below nvec) of a row held in
// shared memory to a base-2 log-sum-exp state.  bf16 takes the batch maximum on
// packed pairs (exact), then one FFMA, one ex2 and one add per element.
template <typename T, int K, int STRIDE>
__device__ __forceinline__ void lse_add_smem(const uint4* sv, int first, int nvec, Lse2& st) {
  constexpr int EPV = Elem<T>::kPerVec;
  const bool full = first + (K - 1) * STRIDE < nvec;  // no vector of this thread is missing
  if (sizeof(T) == 2) {
    uint4 u[K];
    __nv_bfloat162 mx = __float2bfloat162_rn(-INFINITY);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int v = first + k * STRIDE;
      if (full || v < nvec) {
        u[k] = sv[v];
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&u[k].x));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&u[k].y));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&u[k].z));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&u[k].w));
      }
    }
    const float bm = fmaxf(__low2float(mx), __high2float(mx)) * kLog2e;  // monotone
    if (bm > st.m) {
      st.s *= ex2(st.m - bm);
      st.m = bm;
    }
    if (st.m != -INFINITY) {
      // packed fp32 pairs (FFMA2, FADD2) and two accumulators, so the sum is
      // not one long chain of dependent adds
      const float2 lg = make_float2(kLog2e, kLog2e), nm = make_float2(-st.m, -st.m);
      float2 acc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int v = first + k * STRIDE;
        if (full || v < nvec) {
          const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 t = __ffma2_rn(make_float2(bf16_lo(w[i]), bf16_hi(w[i])), lg, nm);
            acc[i & 1] = __fadd2_rn(acc[i & 1], make_float2(ex2(t.x), ex2(t.y)));
          }
        }
      }
      const float2 a2 = __fadd2_rn(acc[0], acc[1]);
      st.s += a2.x + a2.y;
    }
  } else {
    float t[K * EPV];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int v = first + k * STRIDE;
      if (full || v < nvec) {
        float x[EPV];
        Elem<T>::unpack(sv[v], x);
#pragma unroll
        for (int e = 0; e < EPV; ++e) t[k * EPV + e] = x[e] * kLog2e;
      } else {
#pragma unroll
        for (int e = 0; e < EPV; ++e) t[k * EPV + e] = -INFINITY;
      }
    }
    st.addk(t);
  }
}

// Per-row constants of dZ = c * (softmax - onehot).  The scale is folded into
// the exponent: c * 2^(t - lse2) = sign(c) * 2^(t - (lse2 - log2|c|)), so each
// element costs one FFMA and one ex2; a negative c flips the sign bits of the
// packed result.
template <typename T>
struct DzRow {
  float c;       // the scale; 0: the row's gradient is zero
  float l2c;     // lse2 - log2|c|
  uint32_t neg;  // sign mask XORed into each packed 32-bit word when c < 0
  __device__ DzRow(float lse2, float c_) : c(c_) {
    l2c = c_ != 0.0f ? lse2 - log2f(fabsf(c_)) : 0.0f;
    neg = c_ < 0.0f ? (sizeof(T) == 2 ? 0x80008000u : 0x80000000u) : 0u;
  }
};

// Writes dZ for K vectors sv[first + k*STRIDE] (those below nvec) to out[v];
// ylocal is the label's element index relative to sv[0] (out of range when the
// label lies elsewhere).  c == 0 writes zeros.
template <typename T, int K, int STRIDE>
__device__ __forceinline__ void dz_from_smem(const uint4* sv, int first, int nvec, int64_t ylocal,
                                             const DzRow<T>& r, uint4* out) {
  constexpr int EPV = Elem<T>::kPerVec;
  const bool full = first + (K - 1) * STRIDE < nvec;
  if (r.c == 0.0f) {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int v = first + k * STRIDE;
      if (full || v < nvec) __stcs(out + v, z);
    }
    return;
  }
  // the vector holding the label, if it is one of this call's
  const int lab_v = (ylocal >= 0 && ylocal < static_cast<int64_t>(nvec) * EPV)
                        ? static_cast<int>(ylocal / EPV)
                        : -1;
  const float2 lg = make_float2(kLog2e, kLog2e), nl = make_float2(-r.l2c, -r.l2c);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int v = first + k * STRIDE;
    if (full || v < nvec) {
      float x[EPV];
      Elem<T>::unpack(sv[v], x);
#pragma unroll
      for (int e = 0; e < EPV; e += 2) {  // packed fp32 pairs (FFMA2)
        const float2 t = __ffma2_rn(make_float2(x[e], x[e + 1]), lg, nl);
        x[e] = ex2(t.x);
        x[e + 1] = ex2(t.y);
      }
      uint4 o;
      if (v != lab_v) {
        o = Elem<T>::pack(x);
        o.x ^= r.neg;
        o.y ^= r.neg;
        o.z ^= r.neg;
        o.w ^= r.neg;
      } else {  // the one-hot label term
        const int e_y = static_cast<int>(ylocal - static_cast<int64_t>(v) * EPV);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          x[e] = r.neg ? -x[e] : x[e];
          if (e == e_y) x[e] -= r.c;
        }
        o = Elem<T>::pack(x);
      }
      __stcs(out + v, o);
    }
  }
}

// A row as the bulk copies see it: the 16-byte blocks that hold any of its
// elements.  A row need not start on a 16-byte boundary (an odd vocabulary, a
// row stride that is not a multiple of 16 bytes, a column slice): its first
// block then starts `head` elements before the row, and its last block may end
// after it.  Those outside elements belong to a neighbouring row (or lie just
// outside the tensor); they are copied, never used and never written.  A
// 16-byte block never straddles a page, so a block that holds one byte of the
// row is mapped memory as a whole.
struct RowSpan {
  const char* a0;  // the first block
  int head;        // elements of the first block before the row (0: aligned)
  int64_t nvec;    // blocks
};

template <typename T>
__device__ __forceinline__ RowSpan row_span(const void* base, int64_t row, int64_t ld, int64_t V) {
  const uintptr_t rs = reinterpret_cast<uintptr_t>(static_cast<const T*>(base) + row * ld);
  const uintptr_t a0 = rs & ~static_cast<uintptr_t>(15);
  const uintptr_t a1 = (rs + static_cast<uintptr_t>(V) * sizeof(T) + 15) &
                       ~static_cast<uintptr_t>(15);
  RowSpan sp;
  sp.a0 = reinterpret_cast<const char*>(a0);
  sp.head = static_cast<int>((rs - a0) / sizeof(T));
  sp.nvec = static_cast<int64_t>((a1 - a0) / 16);
  return sp;
}

// Elements [lo, hi) of one 16-byte block (a row's first or last block, the
// rest belonging to other rows) added to a base-2 log-sum-exp state.
template <typename T>
__device__ __forceinline__ void lse_add_part(const uint4& v, int lo, int hi, Lse2& st) {
  float x[Elem<T>::kPerVec];
  Elem<T>::unpack(v, x);
#pragma unroll
  for (int e = 0; e < Elem<T>::kPerVec; ++e) {  // unrolled: x stays in registers
    const float t = x[e] * kLog2e;
    if (e >= lo && e < hi && t != -INFINITY) st.add1(t);
  }
}

// dZ of elements [lo, hi) of one 16-byte block, stored one by one to
// out[lo..hi) (the block's other elements belong to other rows); e_y: the
// label's position in the block, or -1.  The same arithmetic as dz_from_smem.
template <typename T>
__device__ __forceinline__ void dz_part(const uint4& v, int lo, int hi, int e_y,
                                        const DzRow<T>& r, T* out) {
  if (r.c == 0.0f) {  // a zero gradient: the block is not read
    for (int e = lo; e < hi; ++e) Elem<T>::store(out + e, 0.0f);
    return;
  }
  float x[Elem<T>::kPerVec];
  Elem<T>::unpack(v, x);
#pragma unroll
  for (int e = 0; e < Elem<T>::kPerVec; ++e) {
    if (e < lo || e >= hi) continue;
    float d = ex2(__fmaf_rn(x[e], kLog2e, -r.l2c));
    if (r.neg) d = -d;
    if (e == e_y) d -= r.c;
    Elem<T>::store(out + e, d);
  }
}

// The blocks [0, nvec) of a piece of a row that starts at row element e0
// (negative in the first piece of a row with a head): the first and the last
// block may hold elements outside [0, V).  Whole blocks are [vb, ve).
struct PieceEdges {
  int vb, ve;
  bool head_part, tail_part;
  __device__ PieceEdges(int64_t e0, int nvec, int64_t V, int epv) {
    head_part = nvec > 0 && e0 < 0;
    tail_part = nvec > 0 && e0 + static_cast<int64_t>(nvec) * epv > V;
    vb = head_part ? 1 : 0;
    ve = tail_part ? nvec - 1 : nvec;
    if (ve < vb) ve = vb;
  }
  __device__ PieceEdges() {}
  // a piece of whole blocks only
  __device__ static PieceEdges whole(int nvec) {
    PieceEdges p;
    p.vb = 0;
    p.ve = nvec;
    p.head_part = p.tail_part = false;
    return p;
  }
};

// The valid element range [lo, hi) of block v of a piece starting at row
// element e0.
__device__ __forceinline__ void block_range(int64_t e0, int v, int64_t V, int epv, int& lo,
                                            int& hi) {
  const int64_t eb = e0 + static_cast<int64_t>(v) * epv;
  lo = eb < 0 ? static_cast<int>(-eb) : 0;
  hi = eb + epv > V ? static_cast<int>(V - eb) : epv;
}

struct StreamArgs {
  const void* logits;
  int64_t N, V, ld;
  const int64_t* labels;
  int64_t ignore_index;
  // forward
  float* lse_out;
  float* loss_rows;
  float* label_logit;
  // backward
  int reduction;
  int64_t num_label_tokens;
  const float* lse_in;
  const int64_t* n_valid;
  const float* grad_loss;
  void* grad;
  int64_t ldg;
  int32_t* status;
  // vocabulary shard (v0 = 0, V_total = V and sh.m_out = nullptr unsharded)
  int64_t v0;
  int64_t V_total;
  ShardOut sh;
};

// kTwoPass (backward only): no saved lse, each row is streamed twice.
// kWhole: every row starts and ends on a 16-byte boundary (the partial-block
// handling is compiled out).
template <typename T, bool kBwd, bool kTwoPass, bool kWhole>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm)
    ce_stream_kernel(const StreamArgs a) {
  constexpr int kVecPerSeg = kSegBytes / 16;
  constexpr int kVecPerThread = kVecPerSeg / kConsumers;  // 8 (32 KB segments)
  extern __shared__ uint8_t ring_raw[];
  __shared__ uint64_t full_bar[kRingStages], empty_bar[kRingStages];
  __shared__ int abort_sh;
  __shared__ float red_m[kConsumerWarps], red_s[kConsumerWarps];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(ring_raw) + 127) & ~static_cast<uintptr_t>(127));
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kRingStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();
  constexpr int EPV = Elem<T>::kPerVec;
  const int seg_elems = kSegBytes / static_cast<int>(sizeof(T));
  auto span = [&](int64_t row) -> RowSpan {
    if (!kWhole) return row_span<T>(a.logits, row, a.ld, a.V);
    RowSpan sp;
    sp.a0 = reinterpret_cast<const char*>(static_cast<const T*>(a.logits) + row * a.ld);
    sp.head = 0;
    sp.nvec = a.V * static_cast<int64_t>(sizeof(T)) / 16;
    return sp;
  };

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      constexpr int npass = (kBwd && kTwoPass) ? 2 : 1;
      for (int64_t row = blockIdx.x; row < a.N && ok; row += gridDim.x) {
        const RowSpan sp = span(row);
        const int64_t cb = sp.nvec * 16;  // bytes copied: the row's blocks
        const int nseg = static_cast<int>((cb + kSegBytes - 1) / kSegBytes);
        for (int it = 0; it < npass * nseg && ok; ++it) {
          const int sg = it % nseg;
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bytes = static_cast<uint32_t>(
              min(static_cast<int64_t>(kSegBytes), cb - static_cast<int64_t>(sg) * kSegBytes));
          // checked builds: the segment lies inside the row's blocks and its
          // stage; a failed check completes the stage without a copy
          if (span_in_range(static_cast<int64_t>(sg) * kSegBytes, bytes, cb, a.status) &&
              smem_in_range(stage * kSegBytes + 128, kSegBytes, a.status)) {
            mbar_arrive_expect_tx(&full_bar[stage], bytes);
            bulk_load(ring + stage * kSegBytes, sp.a0 + static_cast<int64_t>(sg) * kSegBytes,
                      bytes, &full_bar[stage]);
          } else {
            mbar_arrive(&full_bar[stage]);
          }
          ++issued;
          if (++stage == kRingStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(a.status, FLCE_ETIMEOUT);
        for (int i = 0; i < kRingStages && i < issued; ++i) {
          if (stage == 0) {
            stage = kRingStages;
            phase ^= 1u;
          }
          --stage;
          const uint64_t t0 = global_ns();
          while (!mbar_try_wait(smem_u32(&full_bar[stage]), phase) &&
                 global_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  float coef = 0.0f;
  if (kBwd) coef = grad_coef(a.reduction, a.num_label_tokens, a.n_valid, a.grad_loss);
  // backward without a saved lse: every row is streamed twice, a reduction
  // pass (as the forward) and then the transform pass
  constexpr int npass = (kBwd && kTwoPass) ? 2 : 1;
  uint32_t stage = 0, phase = 0;
  for (int64_t row = blockIdx.x; row < a.N; row += gridDim.x) {
    const int64_t yg = a.labels[row];
    const bool valid = (yg != a.ignore_index) && label_ok(yg, a.V_total);
    const int64_t y = valid ? yg - a.v0 : -1;  // label column within this shard (or none)
    float c = 0.0f, lse2 = 0.0f;
    if (kBwd) {
      c = valid ? coef : 0.0f;
      if (!kTwoPass) lse2 = a.lse_in[row] * kLog2e;
    }
    const RowSpan sp = span(row);
    const int64_t cb = sp.nvec * 16;
    const int nseg = static_cast<int>((cb + kSegBytes - 1) / kSegBytes);
    // the output row: same offset within its first block as the input row
    T* out_row = kBwd ? static_cast<T*>(a.grad) + row * a.ldg : nullptr;
    uint4* out_blk = kBwd ? reinterpret_cast<uint4*>(reinterpret_cast<uintptr_t>(out_row) &
                                                     ~static_cast<uintptr_t>(15))
                          : nullptr;
    for (int pass = 0; pass < npass; ++pass) {
      const bool reduce_pass = !kBwd || pass + 1 < npass;
      Lse2 st;
      for (int sg = 0; sg < nseg; ++sg) {
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&full_bar[stage], phase, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const int nvec = static_cast<int>(
            min(static_cast<int64_t>(kSegBytes), cb - static_cast<int64_t>(sg) * kSegBytes) / 16);
        // checked builds: the segment's blocks lie inside the row's blocks
        if (ok && span_in_range(static_cast<int64_t>(sg) * (kSegBytes / 16), nvec, sp.nvec,
                                a.status)) {
          const uint4* sv = reinterpret_cast<const uint4*>(ring + stage * kSegBytes);
          // row element of the segment's first block element
          const int64_t e0 = static_cast<int64_t>(sg) * seg_elems - sp.head;
          const PieceEdges pe = kWhole ? PieceEdges::whole(nvec) : PieceEdges(e0, nvec, a.V, EPV);
          const bool one = pe.head_part && pe.tail_part && nvec == 1;
          if (reduce_pass) {
            lse_add_smem<T, kVecPerThread, kConsumers>(sv + pe.vb, tid, pe.ve - pe.vb, st);
            int lo, hi;
            if (pe.head_part && tid == 0) {
              block_range(e0, 0, a.V, EPV, lo, hi);
              lse_add_part<T>(sv[0], lo, hi, st);
            }
            if (pe.tail_part && !one && tid == kConsumers - 1) {
              block_range(e0, nvec - 1, a.V, EPV, lo, hi);
              lse_add_part<T>(sv[nvec - 1], lo, hi, st);
            }
          } else {
            const DzRow<T> dr(lse2, c);
            const int64_t yb = e0 + static_cast<int64_t>(pe.vb) * EPV;  // row element of sv[vb]
            dz_from_smem<T, kVecPerThread, kConsumers>(
                sv + pe.vb, tid, pe.ve - pe.vb, y >= 0 ? y - yb : -1, dr,
                out_blk + static_cast<int64_t>(sg) * (kSegBytes / 16) + pe.vb);
            int lo, hi;
            if (pe.head_part && tid == 0) {
              block_range(e0, 0, a.V, EPV, lo, hi);
              dz_part<T>(sv[0], lo, hi, (y >= e0 && y < e0 + EPV) ? static_cast<int>(y - e0) : -1,
                         dr, out_row + e0);
            }
            if (pe.tail_part && !one && tid == kConsumers - 1) {
              const int64_t el = e0 + static_cast<int64_t>(nvec - 1) * EPV;
              block_range(e0, nvec - 1, a.V, EPV, lo, hi);
              dz_part<T>(sv[nvec - 1], lo, hi,
                         (y >= el && y < el + EPV) ? static_cast<int>(y - el) : -1, dr,
                         out_row + el);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (++stage == kRingStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!reduce_pass) continue;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, st.m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, st.s, o);
        st.merge(m2, s2);
      }
      if (lane == 0) {
        red_m[warp] = st.m;
        red_s[warp] = st.s;
      }
      named_barrier(1, kConsumers);
      if (kBwd) {
        // every consumer merges the warp states itself (same order, same lse)
        Lse2 all;
        for (int w = 0; w < kConsumerWarps; ++w) all.merge(red_m[w], red_s[w]);
        lse2 = all.m + log2f(all.s);
      } else if (tid == 0) {
        Lse2 all;
        for (int w = 0; w < kConsumerWarps; ++w) all.merge(red_m[w], red_s[w]);
        const T* prow = static_cast<const T*>(a.logits) + row * a.ld;
        if (a.sh.m_out != nullptr) {
          a.sh.write(row, all.m, all.s, yg, a.ignore_index, a.V, prow, a.status);
        } else {
          const float lse = all.m * kLn2 + logf(all.s);
          a.lse_out[row] = lse;
          float li = 0.0f, zy = NAN;
          if (yg != a.ignore_index) {
            if (valid) {
              zy = Elem<T>::load(prow + y);
              li = lse - zy;
            } else {
              set_status(a.status, FLCE_ELABEL);
            }
          }
          a.loss_rows[row] = li;
          if (a.label_logit != nullptr) a.label_logit[row] = zy;
        }
      }
      named_barrier(1, kConsumers);  // red_* is free for the next row
    }
  }
}

template <typename T, bool kBwd, bool kTwoPass, bool kWhole>
static int launch_stream_k(const StreamArgs& a, cudaStream_t s) {
  auto kern = ce_stream_kernel<T, kBwd, kTwoPass, kWhole>;
  static std::atomic<uint64_t> done{0};  // devices whose smem limit is raised
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const uint64_t bit = 1ull << (dev & 63);
  int rc = FLCE_OK;
  if (!(done.load() & bit)) {
    rc = cuda_status(
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem),
        "cudaFuncSetAttribute(ce_stream_kernel)");
    if (rc != FLCE_OK) return rc;
    done.fetch_or(bit);
  }
  const int64_t g = static_cast<int64_t>(sm_count()) * kStreamCtasPerSm;
  const int grid = static_cast<int>(a.N < g ? a.N : g);
  kern<<<grid, kStreamThreads, kStreamSmem, s>>>(a);
  return launch_status(kBwd ? "ce_stream_kernel<bwd> launch" : "ce_stream_kernel<fwd> launch");
}

// Rows that all start and end on 16-byte boundaries take the instance without
// partial-block handling.  (The backward's gradient rows sit at the same
// offsets as the logits rows: the callers check that.)
template <typename T, bool kBwd, bool kTwoPass = false>
static int launch_stream(const StreamArgs& a, cudaStream_t s) {
  const bool whole = reinterpret_cast<uintptr_t>(a.logits) % 16 == 0 &&
                     (a.ld * static_cast<int64_t>(sizeof(T))) % 16 == 0 &&
                     (a.V * static_cast<int64_t>(sizeof(T))) % 16 == 0;
  return whole ? launch_stream_k<T, kBwd, kTwoPass, true>(a, s)
               : launch_stream_k<T, kBwd, kTwoPass, false>(a, s);
}

// ------------------------------ backward without a saved lse: resident rows
//
// The strict "keep only the logits and the labels" backward: the lse is not
// saved, so it has to be formed again before the gradient.  Streaming each row
// twice costs a second read of the logits; instead a row is split over a
// cluster of P CTAs (P = 1, 2, 4 or 8, the fewest whose slices fit kResBuf
// bytes: a bf16 row of V = 128256, 250.5 KiB, in four slices of 62.6 KiB) that
// hold it in shared memory.  Each CTA copies its slice in once (cp.async.bulk,
// 8 KB per mbarrier so the reduction starts on the first piece), reduces it to
// a base-2 (m, s) pair and sends the pair to the other CTAs with st.async
// (8 bytes that complete on the receiver's mbarrier: no cluster-wide barrier
// per row); every CTA merges the P pairs in rank order (so all CTAs of the
// cluster hold the same lse) and writes its slice of dZ from shared memory.
// The logits are read from HBM once, as when the lse is saved.  Rows with a
// zero gradient (ignored labels, or a zero coefficient) are written as zeros
// without being read.  The fused mode (forward and backward in one call)
// also writes each row's loss, from the CTA whose slice holds the label's
// logit, and its lse; it reads every row with a valid label, also when the
// coefficient is zero, since the loss still needs the row.
//
// Measured alternatives on GB300 ([16384, 128256] bf16): two slice buffers
// per CTA (the next row copied in, or a row pipeline that lets the CTAs of a
// cluster drift apart by a row) need twice the CTAs per row and were 15-30%
// slower; one barrier.cluster per row instead of st.async 5% slower; streaming
// each row twice through the ring 25% slower (about even with L2 evict_last /
// evict_first hints at 2 CTAs per SM); copying the next row into each pair of
// segments as soon as its dZ is written (same shared memory) 0.3% faster, not
// worth its bookkeeping.
#ifndef FLCE_CE_RES_BUF
#define FLCE_CE_RES_BUF 65536
#endif
constexpr int kResThreads = 256;
constexpr int kResWarps = kResThreads / 32;
constexpr int kResSeg = 8192;
constexpr int kResSegVec = kResSeg / 16;
constexpr int kResBuf = FLCE_CE_RES_BUF;  // shared-memory bytes for a slice
constexpr int kResMaxSegs = (kResBuf + kResSeg - 1) / kResSeg;
constexpr int kResMaxCluster = 8;
static_assert(kResBuf % 256 == 0 && kResSegVec % kResThreads == 0, "whole vectors per thread");

struct ResArgs {
  const void* logits;
  int64_t N, V, ld;
  const int64_t* labels;
  int64_t ignore_index;
  int reduction;
  int64_t num_label_tokens;
  const int64_t* n_valid;
  const float* grad_loss;
  void* grad;
  int64_t ldg;
  int32_t* status;
  int64_t slice_vec;  // 16-byte vectors per CTA slice (the last slice may be shorter)
  // forward and backward in one pass (ce_logits_fwd_bwd): per-row losses and
  // lse are written too, and every row with a valid label is read, also when
  // its gradient is zero.  loss_rows == nullptr: the backward alone.
  float* loss_rows;
  float* lse_out;  // may be null
};

// kWhole: every row starts and ends on a 16-byte boundary (no partial blocks;
// the edge handling is compiled out).
template <typename T, bool kWhole>
__global__ void __launch_bounds__(kResThreads, 3) ce_bwd_resident_kernel(const ResArgs a) {
  constexpr int EPV = Elem<T>::kPerVec;
  extern __shared__ uint8_t res_raw[];
  __shared__ uint64_t bar[kResMaxSegs];
  // the cluster's (m, s) pairs of a copied row, by rank; copied row k uses slot
  // k % 2, whose barrier completes when the other P - 1 pairs have landed.  Two
  // slots suffice: a CTA sends row k's pair only after it has all pairs of row
  // k - 1, and every CTA reads a row's pairs before it sends the next pair.
  __shared__ __align__(8) float2 pairs[2][kResMaxCluster];
  __shared__ uint64_t xbar[2];
  __shared__ float red_m[kResWarps], red_s[kResWarps];
  __shared__ float lse2_sh;
  __shared__ int abort_sh;
  __shared__ int xbroken_sh;  // set (by thread 0) when an exchange wait timed out
  uint4* buf = reinterpret_cast<uint4*>(
      (reinterpret_cast<uintptr_t>(res_raw) + 127) & ~static_cast<uintptr_t>(127));
  volatile int* abort_flag = &abort_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t P = cluster_nctarank();
  const int64_t nclusters = gridDim.x / P;
  auto span = [&](int64_t r) -> RowSpan {
    if (!kWhole) return row_span<T>(a.logits, r, a.ld, a.V);
    RowSpan sp;
    sp.a0 = reinterpret_cast<const char*>(static_cast<const T*>(a.logits) + r * a.ld);
    sp.head = 0;
    sp.nvec = a.V * static_cast<int64_t>(sizeof(T)) / 16;
    return sp;
  };
  auto edges = [&](int64_t e0, int n) -> PieceEdges {
    return kWhole ? PieceEdges::whole(n) : PieceEdges(e0, n, a.V, EPV);
  };
  // this CTA's slice of a row: blocks [v_lo, v_lo + nv) of the row's 16-byte
  // blocks (rows that start at different offsets within a block can differ by
  // one block)
  auto slice = [&](const RowSpan& sp, int64_t& v_lo, int& nv) {
    v_lo = min(sp.nvec, static_cast<int64_t>(rank) * a.slice_vec);
    nv = static_cast<int>(min(sp.nvec, v_lo + a.slice_vec) - v_lo);
  };
  if (tid == 0) {
    for (int i = 0; i < kResMaxSegs; ++i) mbar_init(&bar[i], 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    // checked builds: a slice fits the shared memory and the barriers of this
    // launch; a failed check skips every copy
    const bool fits =
        in_range(rank, kResMaxCluster, a.status) &&
        span_in_range(0, (a.slice_vec + kResSegVec - 1) / kResSegVec, kResMaxSegs + 1,
                      a.status) &&
        smem_in_range(128, (a.slice_vec + 7) / 8 * 8 * 16, a.status);
    abort_sh = fits ? 0 : 1;
    xbroken_sh = 0;
    fence_barrier_init();
  }
  // the exchange barriers must be initialised in every CTA before any pair is sent
  cluster_sync();
  const float coef = grad_coef(a.reduction, a.num_label_tokens, a.n_valid, a.grad_loss);
  const bool fused = a.loss_rows != nullptr;
  const int64_t first = blockIdx.x / P;

  // Writes this CTA's part of row r of dZ: whole blocks with 16-byte stores,
  // the row's first and last block (shared with other rows) element by
  // element.  sv: the slice in shared memory (unused when dr.c == 0).
  auto write_dz = [&](int64_t r, const RowSpan& sp, int64_t v_lo, int nv, int64_t y,
                      const DzRow<T>& dr) {
    T* out_row = static_cast<T*>(a.grad) + r * a.ldg;
    uint4* ob = reinterpret_cast<uint4*>(reinterpret_cast<uintptr_t>(out_row) &
                                         ~static_cast<uintptr_t>(15)) +
                v_lo;
    const int64_t e0 = v_lo * EPV - sp.head;  // row element of the slice's first block
    const PieceEdges pe = edges(e0, nv);
    const int64_t yb = e0 + static_cast<int64_t>(pe.vb) * EPV;
    const int64_t ylocal = y >= 0 ? y - yb : -1;
    for (int v0 = 0; v0 < pe.ve - pe.vb; v0 += 4 * kResThreads)
      dz_from_smem<T, 4, kResThreads>(buf + pe.vb, v0 + tid, pe.ve - pe.vb, ylocal, dr,
                                      ob + pe.vb);
    int lo, hi;
    if (pe.head_part && tid == 0) {
      block_range(e0, 0, a.V, EPV, lo, hi);
      dz_part<T>(buf[0], lo, hi, (y >= e0 && y < e0 + EPV) ? static_cast<int>(y - e0) : -1, dr,
                 out_row + e0);
    }
    if (pe.tail_part && !(pe.head_part && nv == 1) && tid == kResThreads - 1) {
      const int64_t el = e0 + static_cast<int64_t>(nv - 1) * EPV;
      block_range(e0, nv - 1, a.V, EPV, lo, hi);
      dz_part<T>(buf[nv - 1], lo, hi, (y >= el && y < el + EPV) ? static_cast<int>(y - el) : -1,
                 dr, out_row + el);
    }
  };

  // Rows of this cluster: first + i * nclusters.  Each warp reads the labels
  // of 32 rows at a time (one per lane) and keeps a bit mask of those that need
  // a copy (a nonzero gradient: the same answer in every thread and every CTA
  // of the cluster); rows with a zero gradient are written as zeros when
  // passed, without being read.
  int64_t win = -32;   // index i of the window's first row
  uint32_t todo = 0u;  // bit t: row win + t exists and is not handed out yet
  uint32_t need = 0u;  // bit t: row win + t needs a copy
  const DzRow<T> zero_dr(0.0f, 0.0f);
  auto next_row = [&]() -> int64_t {
    while (true) {
      if (todo == 0u) {
        win += 32;
        if (first + win * nclusters >= a.N) return a.N;
        const int64_t r = first + (win + lane) * nclusters;
        bool nd = false;
        if (r < a.N) {
          const int64_t yr = __ldg(a.labels + r);
          nd = (fused || coef != 0.0f) && yr != a.ignore_index && label_ok(yr, a.V);
        }
        todo = __ballot_sync(0xffffffffu, r < a.N);
        need = __ballot_sync(0xffffffffu, nd);
      }
      const int t = __ffs(todo) - 1;
      todo &= todo - 1u;
      const int64_t r = first + (win + t) * nclusters;
      if ((need >> t) & 1u) return r;
      const RowSpan sp = span(r);
      int64_t v_lo;
      int nv;
      slice(sp, v_lo, nv);
      write_dz(r, sp, v_lo, nv, -1, zero_dr);
      if (fused && rank == 0 && tid == 0) {  // an ignored (or out-of-range) label: no loss
        const int64_t yr = __ldg(a.labels + r);
        if (yr != a.ignore_index) set_status(a.status, FLCE_ELABEL);
        a.loss_rows[r] = 0.0f;
        if (a.lse_out != nullptr) a.lse_out[r] = NAN;
      }
    }
  };

  uint32_t par = 0u;         // bit sg: parity of bar[sg]'s current phase
  uint32_t issued = 0u;      // thread 0: segments with a copy issued
  uint32_t issued_par = 0u;  // thread 0: bit sg, the phase parity of that copy
  uint32_t k = 0;            // copied rows so far
  for (int64_t row = next_row(); row < a.N; row = next_row(), ++k) {
    const int64_t y = __ldg(a.labels + row);
    const RowSpan sp = span(row);
    int64_t v_lo;
    int nv;
    slice(sp, v_lo, nv);
    const int nseg = (nv + kResSegVec - 1) / kResSegVec;
    const int64_t e0 = v_lo * EPV - sp.head;  // row element of the slice's first block
    if (tid == 0 && !*abort_flag) {
      // checked builds: the slice lies inside the row's blocks
      if (!span_in_range(v_lo, nv, sp.nvec, a.status) ||
          !span_in_range(0, nseg, kResMaxSegs + 1, a.status)) {
        *abort_flag = 1;
      } else {
        const char* src = sp.a0 + v_lo * 16;
        for (int sg = 0; sg < nseg; ++sg) {
          const uint32_t bytes =
              static_cast<uint32_t>(min(kResSegVec, nv - sg * kResSegVec)) * 16u;
          mbar_arrive_expect_tx(&bar[sg], bytes);
          bulk_load(buf + sg * kResSegVec, src + static_cast<int64_t>(sg) * kResSeg, bytes,
                    &bar[sg]);
          issued |= 1u << sg;
          issued_par = (issued_par & ~(1u << sg)) | (par & (1u << sg));
        }
      }
    }
    // reduction of the slice, piece by piece as the copies land
    Lse2 st;
    for (int sg = 0; sg < nseg; ++sg) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&bar[sg], (par >> sg) & 1u, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          set_status(a.status, FLCE_ETIMEOUT);
        }
        break;
      }
      const int cnt = min(kResSegVec, nv - sg * kResSegVec);
      const int64_t es0 = e0 + static_cast<int64_t>(sg) * kResSegVec * EPV;
      const PieceEdges pe = edges(es0, cnt);
      const uint4* sv = buf + sg * kResSegVec;
      lse_add_smem<T, kResSegVec / kResThreads, kResThreads>(sv + pe.vb, tid, pe.ve - pe.vb, st);
      int lo, hi;
      if (pe.head_part && tid == 0) {
        block_range(es0, 0, a.V, EPV, lo, hi);
        lse_add_part<T>(sv[0], lo, hi, st);
      }
      if (pe.tail_part && !(pe.head_part && cnt == 1) && tid == kResThreads - 1) {
        block_range(es0, cnt - 1, a.V, EPV, lo, hi);
        lse_add_part<T>(sv[cnt - 1], lo, hi, st);
      }
    }
    par ^= (1u << nseg) - 1u;  // the segments this row used moved to their next phase
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, st.m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, st.s, o);
      st.merge(m2, s2);
    }
    if (lane == 0) {
      red_m[warp] = st.m;
      red_s[warp] = st.s;
    }
    __syncthreads();
    // Exchange of the slices' (m, s) pairs.  After a copy timed out it goes on
    // (with meaningless values) so that no CTA waits for a pair in vain; only
    // an exchange that itself timed out ends the exchanges.
    const int j = static_cast<int>(k & 1u);
    if (warp == 0) {
      if (lane == 0) {
        Lse2 all;
        for (int w = 0; w < kResWarps; ++w) all.merge(red_m[w], red_s[w]);
        pairs[j][rank] = make_float2(all.m, all.s);
        if (P > 1 && !xbroken_sh) {
          mbar_arrive_expect_tx(&xbar[j], (P - 1) * 8u);
          const uint32_t src = smem_u32(&pairs[j][rank]);
          const uint32_t xb = smem_u32(&xbar[j]);
          for (uint32_t q = 0; q < P; ++q)
            if (q != rank) st_async_f32x2(mapa_shared(src, q), all.m, all.s, mapa_shared(xb, q));
        }
      }
      __syncwarp();
      if (P > 1 && !xbroken_sh) {
        // every lane of the warp waits (acquire) before it reads the pairs
        const bool got = mbar_wait(&xbar[j], (k >> 1) & 1u, nullptr, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got) && lane == 0) {
          xbroken_sh = 1;
          *abort_flag = 1;
          set_status(a.status, FLCE_ETIMEOUT);
        }
      }
      float m = -INFINITY, sp2 = 0.0f;
      if (lane < static_cast<int>(P)) {
        const float2 pr = pairs[j][lane];
        m = pr.x;
        sp2 = pr.y;
      }
      Lse2 all;
      for (int q = 0; q < static_cast<int>(P); ++q)
        all.merge(__shfl_sync(0xffffffffu, m, q), __shfl_sync(0xffffffffu, sp2, q));
      if (lane == 0) lse2_sh = all.m + log2f(all.s);
    }
    __syncthreads();
    const float lse2 = lse2_sh;
    if (fused && tid == 0) {
      // the row's loss, from the CTA whose slice holds the label's logit
      const float lse = lse2 * kLn2;
      const int64_t yl = y - e0;  // the label's element within the slice
      if (yl >= 0 && yl < static_cast<int64_t>(nv) * EPV)
        a.loss_rows[row] = lse - Elem<T>::load(reinterpret_cast<const T*>(buf) + yl);
      if (rank == 0 && a.lse_out != nullptr) a.lse_out[row] = lse;
    }
    if (!*abort_flag) write_dz(row, sp, v_lo, nv, y, DzRow<T>(lse2, coef));
    __syncthreads();  // the slice buffer and lse2_sh are free again
  }
  // no CTA leaves while a peer may still be running
  cluster_sync();
  if (tid == 0 && *abort_flag) {
    // let this CTA's copies in flight land before its shared memory is released
    for (int sg = 0; sg < kResMaxSegs; ++sg) {
      if (!((issued >> sg) & 1u)) continue;
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(smem_u32(&bar[sg]), (issued_par >> sg) & 1u) &&
             global_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
}

struct ResCacheEntry {
  int dev, P, es;
  size_t smem;
  bool whole;
  int clusters;
};

// Launches ce_bwd_resident_kernel on clusters of P CTAs (a.slice_vec set);
// returns 1 (nothing launched) when no cluster of that size can be resident.
template <typename T, bool kWhole>
static int launch_resident_k(ResArgs a, int P, cudaStream_t s) {
  const size_t smem = static_cast<size_t>((a.slice_vec + 7) / 8 * 8) * 16 + 128;
  auto kern = ce_bwd_resident_kernel<T, kWhole>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  static std::atomic<uint64_t> raised{0};
  const uint64_t bit = 1ull << (dev & 63);
  if (!(raised.load() & bit)) {
    const int rc = cuda_status(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    kResBuf + 128),
                               "cudaFuncSetAttribute(ce_bwd_resident_kernel)");
    if (rc != FLCE_OK) return rc;
    raised.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(P);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(P), 1, 1);
  cfg.blockDim = dim3(kResThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = P > 1 ? 1 : 0;  // P == 1: a plain launch (each CTA is its own cluster)
  // resident clusters for this (device, P, dtype, shared memory), cached
  static std::mutex mu;
  static std::vector<ResCacheEntry> cache;
  int clusters = -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const auto& e : cache)
      if (e.dev == dev && e.P == P && e.es == static_cast<int>(sizeof(T)) && e.smem == smem &&
          e.whole == kWhole)
        clusters = e.clusters;
  }
  if (clusters < 0) {
    int rc;
    if (P > 1) {
      rc = cuda_status(cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg),
                       "cudaOccupancyMaxActiveClusters(ce_bwd_resident_kernel)");
    } else {
      int per_sm = 0;
      rc = cuda_status(
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kResThreads, smem),
          "cudaOccupancyMaxActiveBlocksPerMultiprocessor(ce_bwd_resident_kernel)");
      clusters = per_sm * sm_count();
    }
    if (rc != FLCE_OK) return rc;
    std::lock_guard<std::mutex> lock(mu);
    cache.push_back({dev, P, static_cast<int>(sizeof(T)), smem, kWhole, clusters});
  }
  if (clusters < 1) return 1;
  const int64_t g = a.N < clusters ? a.N : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(g * P), 1, 1);
  return cuda_status(cudaLaunchKernelEx(&cfg, kern, a), "cudaLaunchKernelEx(ce_bwd_resident_kernel)");
}

// Launches ce_bwd_resident_kernel.  Returns 1 (nothing launched) when a row
// does not fit a cluster of kResMaxCluster slices or no cluster of that size
// can be resident.
template <typename T>
static int launch_resident(ResArgs a, cudaStream_t s) {
  // 16-byte blocks of the longest row: one more than the row's own length
  // when rows may start inside a block
  const int64_t bytes = a.V * static_cast<int64_t>(sizeof(T));
  const bool rows_aligned = reinterpret_cast<uintptr_t>(a.logits) % 16 == 0 &&
                            (a.ld * static_cast<int64_t>(sizeof(T))) % 16 == 0;
  const int64_t nvec_row = (bytes + 15) / 16 + (rows_aligned ? 0 : 1);
  int P = 1;  // the fewest CTAs whose slices fit kResBuf bytes (128-byte aligned)
  while (P <= kResMaxCluster && ((nvec_row + P - 1) / P + 7) / 8 * 8 * 16 > kResBuf) P *= 2;
  if (P > kResMaxCluster) return 1;
  a.slice_vec = (nvec_row + P - 1) / P;
  return rows_aligned && bytes % 16 == 0 ? launch_resident_k<T, true>(a, P, s)
                                         : launch_resident_k<T, false>(a, P, s);
}

// The bulk-copy kernels copy whole 16-byte blocks and write the gradient
// block by block at the same positions, so every gradient row must start at
// the same offset within its block as its logits row (in place, or two
// buffers whose starts and row strides agree modulo 16 bytes).
static bool rows_alike(const void* x, int64_t ld, const void* g, int64_t ldg, size_t es) {
  return (reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(g)) % 16 == 0 &&
         ((ld - ldg) * static_cast<int64_t>(es)) % 16 == 0;
}

// ------------------------------------------------------------------ host side

static thread_local char g_last_error[320] = "no CUDA error recorded";

void record_cuda_error(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
           static_cast<int>(e));
}

static std::mutex g_sm_mutex;
static std::vector<int> g_sm_counts;

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(g_sm_mutex);
  if (static_cast<int>(g_sm_counts.size()) <= dev) g_sm_counts.resize(dev + 1, 0);
  if (g_sm_counts[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_counts[dev] = n > 0 ? n : 1;
  }
  return g_sm_counts[dev];
}

}  // namespace flce

using namespace flce;

extern "C" const char* flce_status_string(int status) {
  switch (status) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_EINVAL: return "FLCE_EINVAL: null pointer or bad argument";
    case FLCE_ESHAPE: return "FLCE_ESHAPE: size out of range or inconsistent";
    case FLCE_EDTYPE: return "FLCE_EDTYPE: unsupported dtype";
    case FLCE_EALIGN: return "FLCE_EALIGN: pointer or row stride misaligned";
    case FLCE_ELABEL: return "FLCE_ELABEL: label outside [0, V) that is not ignore_index";
    case FLCE_EWORKSPACE: return "FLCE_EWORKSPACE: workspace missing or too small";
    case FLCE_ECUDA: return "FLCE_ECUDA: CUDA call failed";
    case FLCE_ENOSUP: return "FLCE_ENOSUP: not supported by this library";
    case FLCE_ETIMEOUT: return "FLCE_ETIMEOUT: a bounded wait inside a kernel gave up";
    case FLCE_EBOUNDS: return "FLCE_EBOUNDS: a device-side index check failed (checked build)";
    default: return "FLCE: unknown status";
  }
}

extern "C" const char* flce_last_cuda_error(void) { return g_last_error; }

extern "C" size_t ce_logits_workspace_bytes(int64_t N, int64_t V) {
  (void)V;
  if (N <= 0) return 0;
  return round_up(static_cast<size_t>(N) * sizeof(float), 256);
}

static int ce_common_checks(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                            const int64_t* labels, int reduction) {
  if (!valid_dtype(dt)) return FLCE_EDTYPE;
  if (!valid_reduction(reduction)) return FLCE_EINVAL;
  if (N < 0 || V < 1 || V >= (int64_t(1) << 31) || ld < V) return FLCE_ESHAPE;
  if (N > 0 && (logits == nullptr || labels == nullptr)) return FLCE_EINVAL;
  if (!aligned(logits, dtype_size(dt)) || !aligned(labels, 8)) return FLCE_EALIGN;
  return FLCE_OK;
}

static int row_grid(int64_t N) {
  const int64_t g = static_cast<int64_t>(sm_count()) * 4;
  return static_cast<int>(N < g ? (N > 0 ? N : 1) : g);
}

// Launches the forward (the bulk-copy ring for every row alignment).
// sh.m_out != nullptr: vocabulary-shard outputs instead of lse / loss rows.
static int ce_fwd_rows(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                       const int64_t* labels, int64_t ignore_index, float* lse, float* rows,
                       float* label_logit, const ShardOut& sh, int32_t* status,
                       cudaStream_t s) {
  if (N == 0) return FLCE_OK;
  StreamArgs a{};
  a.logits = logits;
  a.N = N;
  a.V = V;
  a.ld = ld;
  a.labels = labels;
  a.ignore_index = ignore_index;
  a.lse_out = lse;
  a.loss_rows = rows;
  a.label_logit = label_logit;
  a.status = status;
  a.v0 = sh.m_out != nullptr ? sh.v0 : 0;
  a.V_total = sh.m_out != nullptr ? sh.V_total : V;
  a.sh = sh;
  return dt == FLCE_BF16 ? launch_stream<__nv_bfloat16, false>(a, s)
                         : launch_stream<float, false>(a, s);
}

extern "C" int ce_logits_fwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                             const int64_t* labels, int64_t ignore_index, int reduction,
                             int64_t num_label_tokens, float* loss, int64_t* n_valid, float* lse,
                             float* loss_rows, float* label_logit, void* ws, size_t ws_bytes,
                             int32_t* status, flce_stream_t stream) {
  int rc = ce_common_checks(logits, dt, N, V, ld, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (loss == nullptr || n_valid == nullptr || status == nullptr) return FLCE_EINVAL;
  if (N > 0 && lse == nullptr) return FLCE_EINVAL;
  float* rows = loss_rows;
  if (rows == nullptr && N > 0) {
    if (ws == nullptr || ws_bytes < ce_logits_workspace_bytes(N, V)) return FLCE_EWORKSPACE;
    if (!aligned(ws, 16)) return FLCE_EALIGN;
    rows = static_cast<float*>(ws);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ShardOut none{};
  rc = ce_fwd_rows(logits, dt, N, V, ld, labels, ignore_index, lse, rows, label_logit, none,
                   status, s);
  if (rc != FLCE_OK) return rc;
  return launch_finalize(rows, labels, N, V, ignore_index, reduction, num_label_tokens, loss,
                         n_valid, s);
}

extern "C" int ce_logits_fwd_shard(const void* logits_shard, int dt, int64_t N, int64_t V_shard,
                                   int64_t ld, int64_t vocab_offset, int64_t V_total,
                                   const int64_t* labels, int64_t ignore_index, float* m_local,
                                   float* s_local, float* zy_local, int32_t* status,
                                   flce_stream_t stream) {
  int rc = ce_common_checks(logits_shard, dt, N, V_shard, ld, labels, FLCE_SUM);
  if (rc != FLCE_OK) return rc;
  if (vocab_offset < 0 || V_total < vocab_offset + V_shard || V_total >= (int64_t(1) << 31))
    return FLCE_ESHAPE;
  if (status == nullptr) return FLCE_EINVAL;
  if (N > 0 && (m_local == nullptr || s_local == nullptr || zy_local == nullptr))
    return FLCE_EINVAL;
  ShardOut sh{m_local, s_local, zy_local, vocab_offset, V_total};
  return ce_fwd_rows(logits_shard, dt, N, V_shard, ld, labels, ignore_index, nullptr, nullptr,
                     nullptr, sh, status, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------- bounded-wait self-test

// Waits, through the same bounded mbarrier wait every pipeline of this library
// uses, on a barrier nothing will ever arrive on; after limit_ns the wait gives
// up and FLCE_ETIMEOUT goes to the status word, as a failed pipeline would
// report it.  The kernel always returns.
__global__ void wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_sh, limit_ns))
    set_status(status, FLCE_ETIMEOUT);
}

extern "C" int flce_wait_selftest(int32_t* status, uint64_t limit_ns, flce_stream_t stream) {
  if (status == nullptr) return FLCE_EINVAL;
  if (limit_ns > 2000000000ull) return FLCE_ESHAPE;
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return launch_status("wait_selftest_kernel launch");
}

// ------------------------------------------------- device-side index checks

__global__ void bounds_selftest_kernel(int32_t* status) {
  const int64_t n = 16;
  // one past the end: the check fails in a checked build; nothing is accessed
  if (in_range(n, n, status)) {
  }
}

extern "C" int flce_device_checks(void) { return kDeviceChecks ? 1 : 0; }

extern "C" int flce_bounds_selftest(int32_t* status, flce_stream_t stream) {
  if (status == nullptr) return FLCE_EINVAL;
  bounds_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return launch_status("bounds_selftest_kernel launch");
}

// ------------------------------------------------- packed-document labels

// labels[b, t] = ignore_index where doc[b, t] == 0 (padding) or where the next
// position belongs to another document (doc[b, t+1] != doc[b, t]) or the row
// ends; doc holds 1, 2, ... per packed document and 0 for padding.
__global__ void __launch_bounds__(256) packed_labels_kernel(int64_t* __restrict__ labels,
                                                            const int64_t* __restrict__ doc,
                                                            int64_t B, int64_t T,
                                                            int64_t ignore_index) {
  const int64_t n = B * T;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i % T;
    const int64_t d = doc[i];
    const bool last = (t == T - 1) || (doc[i + 1] != d);
    if (d == 0 || last) labels[i] = ignore_index;
  }
}

extern "C" int flce_mask_packed_labels(int64_t* labels, const int64_t* doc_ids, int64_t B,
                                       int64_t T, int64_t ignore_index, flce_stream_t stream) {
  if (B < 0 || T < 0) return FLCE_ESHAPE;
  if (B == 0 || T == 0) return FLCE_OK;
  if (labels == nullptr || doc_ids == nullptr) return FLCE_EINVAL;
  if (!aligned(labels, 8) || !aligned(doc_ids, 8)) return FLCE_EALIGN;
  const int64_t n = B * T;
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, sm_count() * 8));
  packed_labels_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      labels, doc_ids, B, T, ignore_index);
  return launch_status("packed_labels_kernel launch");
}

// ------------------------------------------------- allocation-free forward

// Per-row loss scratch of ce_logits_fwd_noalloc.  Every GPU that loads the
// library holds this array (4 MiB) until the process exits.  All calls share it.
static __device__ __align__(256) float g_noalloc_rows[CE_LOGITS_NOALLOC_MAX_ROWS];

// The address is cached per device together with the id of the context it was
// looked up in: after a cudaDeviceReset (or any other end of the device's
// primary context) the process runs in a new context, whose id differs, and
// the address is looked up again there.
struct NoallocAddr {
  unsigned long long ctx_id = 0;
  float* ptr = nullptr;
};
static std::mutex g_noalloc_mutex;
static std::vector<NoallocAddr> g_noalloc_addr;  // per device id

typedef CUresult (*NoallocCtxGetCurrentFn)(CUcontext*);
typedef CUresult (*NoallocCtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
static Fn noalloc_driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Id of the context current on the calling thread (binding the current
// device's primary context first if none is), 0 if the driver cannot say.
static int noalloc_context_id(int dev, unsigned long long* id) {
  static const NoallocCtxGetCurrentFn get =
      noalloc_driver_fn<NoallocCtxGetCurrentFn>("cuCtxGetCurrent");
  static const NoallocCtxGetIdFn get_id = noalloc_driver_fn<NoallocCtxGetIdFn>("cuCtxGetId");
  *id = 0;
  if (get == nullptr || get_id == nullptr) return FLCE_OK;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    int rc = cuda_status(cudaSetDevice(dev), "cudaSetDevice");
    if (rc != FLCE_OK) return rc;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return FLCE_OK;
  }
  unsigned long long v = 0;
  if (get_id(ctx, &v) == CUDA_SUCCESS) *id = v;
  return FLCE_OK;
}

// Device address of g_noalloc_rows on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up
// with the device current (once per device and context) and cached.
static int noalloc_scratch(float** out) {
  int dev = 0;
  int rc = cuda_status(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc != FLCE_OK) return rc;
  unsigned long long ctx_id = 0;
  rc = noalloc_context_id(dev, &ctx_id);
  if (rc != FLCE_OK) return rc;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (static_cast<int>(g_noalloc_addr.size()) <= dev) g_noalloc_addr.resize(dev + 1);
  NoallocAddr& a = g_noalloc_addr[dev];
  if (a.ptr == nullptr || a.ctx_id != ctx_id) {
    void* p = nullptr;
    rc = cuda_status(cudaGetSymbolAddress(&p, g_noalloc_rows), "cudaGetSymbolAddress");
    if (rc != FLCE_OK) return rc;
    a.ptr = static_cast<float*>(p);
    a.ctx_id = ctx_id;
  }
  *out = a.ptr;
  return FLCE_OK;
}

extern "C" int ce_logits_fwd_noalloc(const void* logits, int dt, int64_t N, int64_t V,
                                     int64_t ld, const int64_t* labels, int64_t ignore_index,
                                     int reduction, int64_t num_label_tokens, float* loss,
                                     int64_t* n_valid, float* lse, int32_t* status,
                                     flce_stream_t stream) {
  int rc = ce_common_checks(logits, dt, N, V, ld, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (N > CE_LOGITS_NOALLOC_MAX_ROWS) return FLCE_ESHAPE;
  if (loss == nullptr || n_valid == nullptr || status == nullptr) return FLCE_EINVAL;
  if (N > 0 && lse == nullptr) return FLCE_EINVAL;
  float* rows = nullptr;
  rc = noalloc_scratch(&rows);
  if (rc != FLCE_OK) return rc;
  // Nothing in the scratch has to start at zero: the row kernel writes the loss
  // of every row 0..N-1 before the finalize kernel reads it.
  return ce_logits_fwd(logits, dt, N, V, ld, labels, ignore_index, reduction, num_label_tokens,
                       loss, n_valid, lse, rows, nullptr, nullptr, 0, status, stream);
}

// The gradient buffer's rules (N > 0): in place it is the logits storage with
// the same row stride; otherwise it must not overlap the logits.
static int grad_buffer_checks(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                              int inplace_grad, const void* grad_logits, int64_t ld_grad) {
  if (grad_logits == nullptr) return FLCE_EINVAL;
  if (inplace_grad != 0 && inplace_grad != 1) return FLCE_EINVAL;
  if (ld_grad < V) return FLCE_ESHAPE;
  if (!aligned(grad_logits, dtype_size(dt))) return FLCE_EALIGN;
  const size_t es = dtype_size(dt);
  const char* a0 = static_cast<const char*>(logits);
  const char* a1 = a0 + ((N - 1) * ld + V) * es;
  const char* b0 = static_cast<const char*>(grad_logits);
  const char* b1 = b0 + ((N - 1) * ld_grad + V) * es;
  if (inplace_grad) {
    if (b0 != a0 || ld_grad != ld) return FLCE_EINVAL;
  } else if (b0 < a1 && a0 < b1) {
    return FLCE_EINVAL;  // out-of-place buffers must not overlap
  }
  return FLCE_OK;
}

// grad_loss may be null only for the library's own calls (g = 1).
static int ce_bwd_entry(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                        int64_t v0, int64_t V_total, const int64_t* labels,
                        int64_t ignore_index, int reduction, int64_t num_label_tokens,
                        const float* lse, const int64_t* n_valid, const float* grad_loss,
                        int inplace_grad, void* grad_logits, int64_t ld_grad, int32_t* status,
                        flce_stream_t stream, bool g_optional = false) {
  int rc = ce_common_checks(logits, dt, N, V, ld, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (v0 < 0 || V_total < v0 + V || V_total >= (int64_t(1) << 31)) return FLCE_ESHAPE;
  if (status == nullptr) return FLCE_EINVAL;
  if (N == 0) return FLCE_OK;
  if (n_valid == nullptr || (grad_loss == nullptr && !g_optional)) return FLCE_EINVAL;
  // no saved lse: only for a whole vocabulary (a shard needs the global lse)
  if (lse == nullptr && (v0 != 0 || V_total != V)) return FLCE_EINVAL;
  rc = grad_buffer_checks(logits, dt, N, V, ld, inplace_grad, grad_logits, ld_grad);
  if (rc != FLCE_OK) return rc;
  const size_t es = dtype_size(dt);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool stream_ok = rows_alike(logits, ld, grad_logits, ld_grad, es);
  if (stream_ok && lse == nullptr) {
    ResArgs r{};
    r.logits = logits;
    r.N = N;
    r.V = V;
    r.ld = ld;
    r.labels = labels;
    r.ignore_index = ignore_index;
    r.reduction = reduction;
    r.num_label_tokens = num_label_tokens;
    r.n_valid = n_valid;
    r.grad_loss = grad_loss;
    r.grad = grad_logits;
    r.ldg = ld_grad;
    r.status = status;
    rc = dt == FLCE_BF16 ? launch_resident<__nv_bfloat16>(r, s) : launch_resident<float>(r, s);
    if (rc != 1) return rc;
    // a row too long for one cluster: streamed twice below
  }
  if (stream_ok) {
    StreamArgs a{};
    a.logits = logits;
    a.N = N;
    a.V = V;
    a.ld = ld;
    a.labels = labels;
    a.ignore_index = ignore_index;
    a.reduction = reduction;
    a.num_label_tokens = num_label_tokens;
    a.lse_in = lse;
    a.n_valid = n_valid;
    a.grad_loss = grad_loss;
    a.grad = grad_logits;
    a.ldg = ld_grad;
    a.status = status;
    a.v0 = v0;
    a.V_total = V_total;
    if (lse == nullptr)
      return dt == FLCE_BF16 ? launch_stream<__nv_bfloat16, true, true>(a, s)
                             : launch_stream<float, true, true>(a, s);
    return dt == FLCE_BF16 ? launch_stream<__nv_bfloat16, true>(a, s)
                           : launch_stream<float, true>(a, s);
  }
  const int grid = row_grid(N);
  if (dt == FLCE_BF16) {
    ce_bwd_rows_kernel<__nv_bfloat16, 512><<<grid, 512, 0, s>>>(
        static_cast<const __nv_bfloat16*>(logits), N, V, ld, labels, ignore_index, reduction,
        num_label_tokens, lse, n_valid, grad_loss, static_cast<__nv_bfloat16*>(grad_logits),
        ld_grad, v0, V_total);
  } else {
    ce_bwd_rows_kernel<float, 512><<<grid, 512, 0, s>>>(
        static_cast<const float*>(logits), N, V, ld, labels, ignore_index, reduction,
        num_label_tokens, lse, n_valid, grad_loss, static_cast<float*>(grad_logits), ld_grad,
        v0, V_total);
  }
  return launch_status("ce_bwd_rows_kernel launch");
}

extern "C" int ce_logits_bwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                             const int64_t* labels, int64_t ignore_index, int reduction,
                             int64_t num_label_tokens, const float* lse, const int64_t* n_valid,
                             const float* grad_loss, int inplace_grad, void* grad_logits,
                             int64_t ld_grad, int32_t* status, flce_stream_t stream) {
  return ce_bwd_entry(logits, dt, N, V, ld, 0, V, labels, ignore_index, reduction,
                      num_label_tokens, lse, n_valid, grad_loss, inplace_grad, grad_logits,
                      ld_grad, status, stream);
}

extern "C" int ce_logits_bwd_shard(const void* logits_shard, int dt, int64_t N, int64_t V_shard,
                                   int64_t ld, int64_t vocab_offset, int64_t V_total,
                                   const int64_t* labels, int64_t ignore_index, int reduction,
                                   int64_t num_label_tokens, const float* lse,
                                   const int64_t* n_valid, const float* grad_loss,
                                   int inplace_grad, void* grad_logits, int64_t ld_grad,
                                   int32_t* status, flce_stream_t stream) {
  return ce_bwd_entry(logits_shard, dt, N, V_shard, ld, vocab_offset, V_total, labels,
                      ignore_index, reduction, num_label_tokens, lse, n_valid, grad_loss,
                      inplace_grad, grad_logits, ld_grad, status, stream);
}

// ------------------------------------------------- forward and backward in one call

extern "C" size_t ce_logits_fwd_bwd_workspace_bytes(int64_t N, int64_t V) {
  if (N < 0 || V < 1) return 0;
  // per-row losses and, for the two-call fallback, a per-row lse
  return 2 * round_up(static_cast<size_t>(N) * 4, 256);
}

extern "C" int ce_logits_fwd_bwd(const void* logits, int dt, int64_t N, int64_t V, int64_t ld,
                                 const int64_t* labels, int64_t ignore_index, int reduction,
                                 int64_t num_label_tokens, const float* grad_loss, float* loss,
                                 int64_t* n_valid, float* lse, int inplace_grad,
                                 void* grad_logits, int64_t ld_grad, void* ws, size_t ws_bytes,
                                 int32_t* status, flce_stream_t stream) {
  int rc = ce_common_checks(logits, dt, N, V, ld, labels, reduction);
  if (rc != FLCE_OK) return rc;
  if (loss == nullptr || n_valid == nullptr || status == nullptr) return FLCE_EINVAL;
  if (N > 0) {
    rc = grad_buffer_checks(logits, dt, N, V, ld, inplace_grad, grad_logits, ld_grad);
    if (rc != FLCE_OK) return rc;
  }
  const size_t need = ce_logits_fwd_bwd_workspace_bytes(N, V);
  if (N > 0 && (ws == nullptr || ws_bytes < need)) return FLCE_EWORKSPACE;
  if (ws != nullptr && !aligned(ws, 16)) return FLCE_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  float* rows = reinterpret_cast<float*>(w);
  float* lse_buf = reinterpret_cast<float*>(w + round_up(static_cast<size_t>(N) * 4, 256));
  const size_t es = dtype_size(dt);
  if (N > 0 && rows_alike(logits, ld, grad_logits, ld_grad, es)) {
    // one pass: the count of valid rows first (the mean's divisor), then each
    // row read once by a row cluster that forms its lse, loss and gradient
    rc = flce_count_valid(labels, N, V, ignore_index, n_valid, stream);
    if (rc != FLCE_OK) return rc;
    ResArgs r{};
    r.logits = logits;
    r.N = N;
    r.V = V;
    r.ld = ld;
    r.labels = labels;
    r.ignore_index = ignore_index;
    r.reduction = reduction;
    r.num_label_tokens = num_label_tokens;
    r.n_valid = n_valid;
    r.grad_loss = grad_loss;  // null: g = 1
    r.grad = grad_logits;
    r.ldg = ld_grad;
    r.status = status;
    r.loss_rows = rows;
    r.lse_out = lse;
    rc = dt == FLCE_BF16 ? launch_resident<__nv_bfloat16>(r, s) : launch_resident<float>(r, s);
    if (rc == FLCE_OK)
      return launch_finalize(rows, labels, N, V, ignore_index, reduction, num_label_tokens, loss,
                             n_valid, s);
    if (rc != 1) return rc;
  }
  // rows that no cluster holds: the forward, then the backward
  float* l = lse != nullptr ? lse : lse_buf;
  // (the per-row losses go to the workspace: ce_logits_fwd needs none of its own)
  rc = ce_logits_fwd(logits, dt, N, V, ld, labels, ignore_index, reduction, num_label_tokens, loss,
                     n_valid, l, rows, nullptr, nullptr, 0, status, stream);
  if (rc != FLCE_OK || N == 0) return rc;
  return ce_bwd_entry(logits, dt, N, V, ld, 0, V, labels, ignore_index, reduction,
                      num_label_tokens, l, n_valid, grad_loss, inplace_grad, grad_logits,
                      ld_grad, status, stream, true);
}
