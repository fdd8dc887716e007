// Persistent tcgen05 GEMM with a pluggable epilogue, for sm_103a.
//
//   acc[m, n] = sum_k A[m, k] * B[n, k]          (fp32 accumulation in TMEM)
//
// A and B are each either K-major (row-major [rows, K]) or MN-major (row-major
// [K, rows]); both come from global memory through TMA with 128-byte swizzle.
// The tile is 128 x BN (BN = 256 or 128) with 128 bytes of K per pipeline
// stage (64 bf16 or 32 fp32 elements).
//
// Warp roles (192 threads):
//   warp 0      TMA producer (one lane): fills the shared-memory ring
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  epilogue: each warp drains the 32 TMEM lanes (tile rows) it
//               may access, 32 columns at a time, and hands the values to
//               Epi::tile.
// The accumulator is double-buffered in TMEM (2 * BN columns), so the
// epilogue of one tile overlaps the main loop of the next.  Tiles are handed
// out statically (tile = blockIdx.x + i * gridDim.x) in a grouped raster
// (group_m M-tiles share each sweep over the N-tiles) for L2 reuse.
//
// Every wait is bounded; on a timeout the kernel records FLCE_ETIMEOUT in the
// status word, stops issuing work, waits (bounded) for work in flight and
// frees its TMEM before returning.
#pragma once

#include "common.cuh"

namespace flce {

constexpr int kBM = 128;
constexpr int kGemmThreads = 192;

template <typename T>
struct MmaTraits;
template <>
struct MmaTraits<__nv_bfloat16> {
  static constexpr uint32_t kFormat = 1;  // bf16 in kind::f16
  static constexpr int kUmmaK = 16;
  __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t i, uint32_t acc) {
    mma_f16(d, a, b, i, acc);
  }
};
template <>
struct MmaTraits<float> {
  static constexpr uint32_t kFormat = 2;  // tf32 in kind::tf32
  static constexpr int kUmmaK = 8;
  __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t i, uint32_t acc) {
    mma_tf32(d, a, b, i, acc);
  }
};

// EW: epilogue warps, 4 (one per TMEM lane quarter) or 8 (two per quarter,
// each draining half of the tile's columns; one stage fewer to make room for
// their staging buffers).
template <typename T, int BN, int EW = 4>
struct GemmGeo {
  static_assert(EW == 4 || EW == 8, "four or eight epilogue warps");
  static constexpr int kEK = 128 / static_cast<int>(sizeof(T));  // K elements per stage
  static constexpr int kStageA = kBM * 128;
  static constexpr int kStageB = BN * 128;
  static constexpr int kStageBytes = kStageA + kStageB;
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr int kTmemCols = 2 * BN;
  // Output staging: two 4 KB buffers per epilogue warp, or one with eight
  // warps (which keeps the fourth stage: at K = 768 the deeper ring took the
  // dZ contraction from 86.1 to 81.8 us, the single buffer costing less)
  static constexpr int kStagingBufs = EW == 8 ? 1 : 2;
  static constexpr int kEpiSmem = EW * kStagingBufs * 4096;
  static constexpr int kSmemBytes =
      kStages * kStageBytes + kEpiSmem + 1024;  // + 1024-byte alignment slack
  static constexpr int kMmaPerStage = 128 / (MmaTraits<T>::kUmmaK * static_cast<int>(sizeof(T)));
  static constexpr int kThreads = 64 + 32 * EW;
};

// Work the epilogue warps do before their first tile, while the producer and
// MMA warps run the first main loops: a small reduction that closes an output
// of the kernels before this one (launches are stream-ordered, so those have
// completed).  Every epilogue warp of the grid takes a fixed share, in a fixed
// order, so the result is the same on every run.
struct EpiPre {
  int kind = 0;                // 0 none, 1 column sums, 2 split-K close
  const float* part = nullptr;
  int nparts = 0;              // 1: partial rows; 2: splits
  int64_t ld = 0;              // 1: row stride; 2: split stride (floats)
  int64_t n = 0;               // 1: columns; 2: output elements / 4
  void* out = nullptr;         // 1: float [n]; 2: bf16 or float [4 n]
  int out_bf16 = 0;            // 2: the output is bf16
  int beta = 0;                // 1: add to the existing out
};

// kind 1: out[v] (+)= sum over s of part[s * ld + v], s in order; kind 2:
// out[4i .. 4i + 3] = sum over splits of part[s * ld + 4i ..], 16-byte loads.
// worker / workers: this warp's index among all epilogue warps of the grid.
__device__ __forceinline__ void epi_pre_run(const EpiPre& q, int worker, int workers, int lane) {
  if (q.kind == 1) {
    for (int64_t c = static_cast<int64_t>(worker) * 32 + lane; c - lane < q.n;
         c += static_cast<int64_t>(workers) * 32) {
      if (c >= q.n) continue;
      float acc = 0.0f;
#pragma unroll 8
      for (int sp = 0; sp < q.nparts; ++sp) acc += q.part[sp * q.ld + c];
      float* o = static_cast<float*>(q.out) + c;
      *o = q.beta ? *o + acc : acc;
    }
  } else if (q.kind == 2) {
    for (int64_t i = static_cast<int64_t>(worker) * 32 + lane; i < q.n;
         i += static_cast<int64_t>(workers) * 32) {
      float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int sp = 0; sp < q.nparts; ++sp) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(q.part + sp * q.ld) + i);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      if (q.out_bf16)
        reinterpret_cast<uint2*>(q.out)[i] =
            make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
      else
        reinterpret_cast<float4*>(q.out)[i] = acc;
    }
  }
}

struct GemmArgs {
  int M, N, K;     // problem size (elements)
  int nMt, nNt, nK;
  int group_m;
  int32_t* status;
  // Split-K (one-CTA kernel only): K blocks are split into k_splits ranges of
  // kb_per_split; split s of M-tile mt is handed to the epilogue as M-tile
  // s * nMt + mt, so each split fills its own row band of the output.
  int k_splits;
  int kb_per_split;
  EpiPre pre;
};

__device__ __forceinline__ void tile_coords(int t, int nMt, int nNt, int group_m, int& mt,
                                            int& nt) {
  const int per_group = group_m * nNt;
  const int g = t / per_group;
  const int first = g * group_m;
  const int gsize = min(group_m, nMt - first);
  const int r = t - g * per_group;
  nt = r / gsize;
  mt = first + (r - nt * gsize);
}

// Loads one operand's share of a stage: `rows` rows starting at row0, K block kb.
template <typename T, bool MN>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                             int rows, int row0, int kb) {
  constexpr int EK = 128 / static_cast<int>(sizeof(T));
  if (!MN) {
    // K-major: one box {EK (K), rows}
    tma_load_2d(dst, map, bar, kb * EK, row0);
  } else {
    // MN-major: rows/EK slabs, each a box {EK (MN), EK (K rows)} of EK*128 bytes
    for (int s = 0; s < rows / EK; ++s)
      tma_load_2d(dst + s * EK * 128, map, bar, row0 + s * EK, kb * EK);
  }
}

// Descriptor of the k-th MMA of a stage for one operand.
template <typename T, bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k) {
  constexpr int EK = 128 / static_cast<int>(sizeof(T));
  constexpr int UK = MmaTraits<T>::kUmmaK;
  if (!MN) {
    // K-major SW128: rows of 128 B, 8-row atoms 1024 B apart; step 32 B along K.
    return smem_desc_sw128(base + k * UK * static_cast<int>(sizeof(T)), 16, 1024);
  } else {
    // MN-major SW128: slabs of EK MN-elements x EK K-rows (EK*128 B apart, the
    // leading byte offset); 8-row K groups 1024 B apart (stride byte offset).
    return smem_desc_sw128(base + k * UK * 128, EK * 128, 1024);
  }
}

// Output staging of one epilogue warp: one or two 4 KB buffers (32 rows x
// 128 B, 1024-byte aligned) written with the 128-byte swizzle the output
// tensor map uses, each then stored (or reduce-added) to global memory by one
// TMA instruction.  Rows and columns outside the tensor are clipped by the TMA.
struct EpiCtx {
  const CUtensorMap* map;
  uint8_t* buf;
  int next;
  int lane;
  int nbuf = 2;  // staging buffers (1 or 2)
  int next_nt = -1;  // the N-tile of this CTA's next tile (-1: none), for prefetches
  int aux = 0, aux_nt = -1;  // an epilogue's own state across tiles

  __device__ void store_slab(const uint4 (&row)[8], int c0, int r0, bool reduce) {
    uint8_t* b = buf + next * 4096;
    if (lane == 0) {  // the buffer's previous store has read it
      if (nbuf == 2)
        bulk_wait_read_le1();
      else
        bulk_wait_read_all();
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(b + lane * 128 + ((j ^ (lane & 7)) << 4)) = row[j];
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        tma_reduce_add_2d(map, b, c0, r0);
      else
        tma_store_2d(map, b, c0, r0);
      bulk_commit();
    }
    next ^= nbuf - 1;
  }

  // Column sums, in row order, of the bf16 slab staged last: lane l sums the
  // 32-bit word at byte 4l of each of the 32 rows, i.e. columns 2l (x) and
  // 2l + 1 (y).  For a fixed row the 32 lanes read 32 distinct banks.
  __device__ float2 last_slab_bf16_column_sums() const {
    const uint8_t* b = buf + ((next ^ 1) & (nbuf - 1)) * 4096;
    const int chunk = lane >> 2, off = (lane & 3) << 2;
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll 8
    for (int r = 0; r < 32; ++r) {
      const uint32_t w =
          *reinterpret_cast<const uint32_t*>(b + r * 128 + ((chunk ^ (r & 7)) << 4) + off);
      acc = __fadd2_rn(acc, make_float2(bf16_lo(w), bf16_hi(w)));
    }
    return acc;
  }

  __device__ void drain() {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};

template <typename T, int BN, bool A_MN, bool B_MN, class Epi, int EW = 4>
__global__ void __launch_bounds__(64 + 32 * EW, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs ga,
                   const typename Epi::Params ep) {
  using G = GemmGeo<T, BN, EW>;
  constexpr int S = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S], accf_bar[2], acce_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf_bar[i], 1);
      mbar_init(&acce_bar[i], EW);
    }
    mbar_init(&drain_bar, 1);
    // checked builds: the stages and staging buffers fit the launch's shared memory
    abort_sh = smem_in_range(0, G::kSmemBytes, ga.status) ? 0 : 1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, G::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int nMtE = ga.nMt * ga.k_splits;  // M-tiles counting every K split
  const int num_tiles = nMtE * ga.nNt;

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(ga.status, FLCE_ETIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mte, nt;
        tile_coords(t, nMtE, ga.nNt, ga.group_m, mte, nt);
        const int split = mte / ga.nMt;
        const int mt = mte - split * ga.nMt;
        const int kb0 = split * ga.kb_per_split;
        const int kb1 = min(ga.nK, kb0 + ga.kb_per_split);
        // checked builds: the tile and its K range lie inside the problem
        if (!in_range(mt, ga.nMt, ga.status) || !in_range(nt, ga.nNt, ga.status) ||
            !span_in_range(kb0, kb1 - kb0, ga.nK, ga.status)) {
          ok = false;
          break;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * G::kStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], G::kStageBytes);
          load_operand<T, A_MN>(sa, &tmA, &full_bar[stage], kBM, mt * kBM, kb);
          load_operand<T, B_MN>(sa + G::kStageA, &tmB, &full_bar[stage], BN, nt * BN, kb);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        fail();
        // let the copies already in flight land before the CTA exits
        for (int i = 0; i < S && i < issued; ++i) {
          if (stage == 0) {
            stage = S;
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
  } else if (warp == 1) {
    if (lane == 0) {
      // ----------------------------------------------------------------- MMA
      constexpr uint32_t idesc = make_idesc(MmaTraits<T>::kFormat, kBM, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        int mte, nt;
        tile_coords(t, nMtE, ga.nNt, ga.group_m, mte, nt);
        const int kb0 = (mte / ga.nMt) * ga.kb_per_split;
        const int kb1 = min(ga.nK, kb0 + ga.kb_per_split);
        if (!mbar_wait(&acce_bar[buf], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * G::kStageBytes);
          const uint32_t sb = sa + G::kStageA;
#pragma unroll
          for (int k = 0; k < G::kMmaPerStage; ++k) {
            MmaTraits<T>::mma(d_tmem, operand_desc<T, A_MN>(sa, k), operand_desc<T, B_MN>(sb, k),
                              idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&empty_bar[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&accf_bar[buf]);
      }
      if (!ok) fail();
      // wait (bounded) until every MMA issued above has finished
      mma_commit(&drain_bar);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(smem_u32(&drain_bar), 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes this warp may access: 32*quad .. +31
    const int row_in_tile = quad * 32 + lane;
    const int half = (warp - 2) >> 2;  // EW == 8: which half of the tile's columns
    EpiCtx ctx;
    ctx.map = &tmC;
    ctx.buf = smem + S * G::kStageBytes + (warp - 2) * G::kStagingBufs * 4096;
    ctx.nbuf = G::kStagingBufs;
    ctx.next = 0;
    ctx.lane = lane;
    epi_pre_run(ga.pre, static_cast<int>(blockIdx.x) * EW + (warp - 2),
                static_cast<int>(gridDim.x) * EW, lane);
    int local = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&accf_bar[buf], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      int mte, nt;
      tile_coords(t, nMtE, ga.nNt, ga.group_m, mte, nt);
      if (t + static_cast<int>(gridDim.x) < num_tiles) {
        int mte2;
        tile_coords(t + static_cast<int>(gridDim.x), nMtE, ga.nNt, ga.group_m, mte2, ctx.next_nt);
      } else {
        ctx.next_nt = -1;
      }
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
      if constexpr (EW == 4)
        Epi::template tile<BN>(ep, mte, nt, row_in_tile, taddr, ctx);
      else
        Epi::template tile_part<BN>(ep, mte, nt, row_in_tile, taddr, ctx, half * (BN / 2),
                                    (half + 1) * (BN / 2));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[buf]);
    }
    ctx.drain();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, G::kTmemCols);
  }
}

}  // namespace flce

// =====================================================================
// CTA-pair variant (bf16): a cluster of two CTAs on two SMs computes one
// 256 x BN tile with tcgen05.mma.cta_group::2.  Each CTA loads its own 128 rows
// of A and its own BN/2 rows of B (so each SM moves half of B through shared
// memory), the leader CTA (rank 0) issues the MMAs for the pair, and each CTA's
// TMEM holds the accumulator rows of its own half.  Stages are 32 KB, so six
// fit beside the epilogue staging buffers.
//
// Synchronisation:
//   full[s]   leader only: one arrive (expect_tx for both CTAs' bytes); both
//             CTAs' TMA loads complete_tx on it (the peer through its
//             shared::cluster address)
//   empty[s]  both CTAs: the leader's MMA commit arrives on both (multicast)
//   accf[b]   both CTAs: accumulator b ready (multicast commit)
//   acce[b]   leader only: 8 arrivals, the epilogue warps of both CTAs
// =====================================================================

namespace flce {

template <int BN>
struct PairGeo {
  static constexpr int kEK = 64;  // bf16 elements per 128-byte row
  static constexpr int kHalfN = BN / 2;
  static constexpr int kStageA = kBM * 128;
  static constexpr int kStageB = kHalfN * 128;
  static constexpr int kStageBytes = kStageA + kStageB;
  static constexpr int kStages = 6;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kEpiSmem = 4 * 2 * 4096;
  static constexpr int kSmemBytes = kStages * kStageBytes + kEpiSmem + 1024;
  static constexpr int kMmaPerStage = 4;
};

template <bool MN>
__device__ __forceinline__ void load_operand_pair(uint8_t* dst, const CUtensorMap* map,
                                                  uint32_t bar_cluster, int rows, int row0,
                                                  int kb) {
  constexpr int EK = 64;
  if (!MN) {
    tma_load_2d_pair(dst, map, bar_cluster, kb * EK, row0);
  } else {
    for (int s = 0; s < rows / EK; ++s)
      tma_load_2d_pair(dst + s * EK * 128, map, bar_cluster, row0 + s * EK, kb * EK);
  }
}

template <int BN, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmArgs ga,
                        const typename Epi::Params ep) {
  using G = PairGeo<BN>;
  using T = __nv_bfloat16;
  constexpr int S = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[S], empty_bar[S], accf_bar[2], acce_bar[2], drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;

  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf_bar[i], 1);
      mbar_init(&acce_bar[i], 8);
    }
    mbar_init(&drain_bar, 1);
    // checked builds: the stages and staging buffers fit the launch's shared memory
    abort_sh = smem_in_range(0, G::kSmemBytes, ga.status) ? 0 : 1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, G::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised; TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  const int cluster_id = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);
  const int num_tiles = ga.nMt * ga.nNt;  // nMt counts 256-row tiles
  const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[0]), 0);
  const uint32_t acce_leader = mapa_shared(smem_u32(&acce_bar[0]), 0);

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(ga.status, FLCE_ETIMEOUT);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = cluster_id; t < num_tiles && ok; t += nclusters) {
        int mt, nt;
        tile_coords(t, ga.nMt, ga.nNt, ga.group_m, mt, nt);
        const int arow = mt * 2 * kBM + static_cast<int>(rank) * kBM;
        const int brow = nt * BN + static_cast<int>(rank) * G::kHalfN;
        // checked builds: the tile lies inside the problem (the same test in both CTAs)
        if (!in_range(mt, ga.nMt, ga.status) || !in_range(nt, ga.nNt, ga.status)) {
          ok = false;
          break;
        }
        for (int kb = 0; kb < ga.nK; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * G::kStageBytes);
          uint8_t* sa = smem + stage * G::kStageBytes;
          const uint32_t fb = full_leader + stage * 8u;
          load_operand_pair<A_MN>(sa, &tmA, fb, kBM, arow, kb);
          load_operand_pair<B_MN>(sa + G::kStageA, &tmB, fb, G::kHalfN, brow, kb);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        fail();
        // copies in flight complete on the leader's barrier; give them time to land
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 20000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // --------------------------------------------------------- MMA (leader)
      constexpr uint32_t idesc = make_idesc(1, 2 * kBM, BN, A_MN, B_MN);
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = cluster_id; t < num_tiles && ok; t += nclusters, ++local) {
        const int buf = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&acce_bar[buf], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < ga.nK; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * G::kStageBytes);
          const uint32_t sb = sa + G::kStageA;
#pragma unroll
          for (int k = 0; k < G::kMmaPerStage; ++k) {
            mma_f16_pair(d_tmem, operand_desc<T, A_MN>(sa, k), operand_desc<T, B_MN>(sb, k),
                         idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&accf_bar[buf], 0x3);
      }
      if (!ok) fail();
      mma_commit_pair(&drain_bar, 0x1);
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(smem_u32(&drain_bar), 0) && global_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    EpiCtx ctx;
    ctx.map = &tmC;
    ctx.buf = smem + S * G::kStageBytes + (warp - 2) * 2 * 4096;
    ctx.next = 0;
    ctx.lane = lane;
    epi_pre_run(ga.pre, static_cast<int>(blockIdx.x) * 4 + (warp - 2),
                static_cast<int>(gridDim.x) * 4, lane);
    int local = 0;
    for (int t = cluster_id; t < num_tiles; t += nclusters, ++local) {
      const int buf = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&accf_bar[buf], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      int mt, nt;
      tile_coords(t, ga.nMt, ga.nNt, ga.group_m, mt, nt);
      if (t + nclusters < num_tiles) {
        int mt2;
        tile_coords(t + nclusters, ga.nMt, ga.nNt, ga.group_m, mt2, ctx.next_nt);
      } else {
        ctx.next_nt = -1;
      }
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(buf * BN);
      // this CTA's half of the 256-row tile is 128-row tile 2*mt + rank
      Epi::template tile<BN>(ep, 2 * mt + static_cast<int>(rank), nt, row_in_tile, taddr, ctx);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&acce_bar[buf]);
        else
          mbar_arrive_cluster(acce_leader + static_cast<uint32_t>(buf) * 8u);
      }
    }
    ctx.drain();
  }

  tc_fence_before();
  cluster_sync();  // both CTAs done with the pair's TMEM and shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, G::kTmemCols);
  }
}

}  // namespace flce
