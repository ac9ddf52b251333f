// Fused, tiled attention forward for sm_103a (GB300).
//
// Computes, per (batch*head, query row i):
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j,   lse_i = ln sum_j exp(scale * q_i . k_j)
// over j in {0..N-1} (or {0..i} when causal), without writing the score matrix to memory.
//
// The method is the tiled loop with an online softmax described in "Android Transformer
// Optimization: Attention and Mobile GPU Bottlenecks" (sections "The Essence of
// FlashAttention: Reordering the Computation" and "A Complete Tile Loop"): query rows are
// cut into tiles, each tile streams the K/V column tiles, keeps a running row max m and
// denominator l, rescales the accumulated O by exp(m_old - m_new) when the max grows, and
// normalises once at the end. The mapping onto GB300 is this file's own:
//
//   * One CTA per SM (persistent), 320 threads = 10 warps:
//       warps 0-3  softmax warpgroup for query tile 0 of the work item (one thread per row)
//       warps 4-7  softmax warpgroup for query tile 1
//       warp  8    tcgen05 MMA issuer (one thread) and TMEM owner
//       warp  9    TMA producer (one thread)
//   * A work item is (batch*head, 256 query rows) = two 128-row query tiles sharing every
//     K/V tile that is loaded. K and V tiles (128 keys x D) stream through a shared-memory
//     ring filled by TMA (128-byte swizzle), synchronised with mbarriers.
//   * S = Q K^T for each query tile goes to its own 128 TMEM columns (fp32). The softmax
//     warpgroup reads its row of S (tcgen05.ld, lane = row), writes P as fp16/bf16 back into
//     the same TMEM columns, and the MMA warp computes O += P V with P read from TMEM.
//     O (fp32, D columns per query tile) stays in TMEM for the whole K/V loop.
//   * The max used in the exponent is only moved when a tile raises the row max by more than
//     2^8; otherwise p = 2^(x - m_used) may exceed 1 (at most 256). O and l always carry the
//     same factor, so the final O / l is unchanged; the rescale of O in TMEM is skipped in
//     most iterations.
//   * Causal: K/V tiles to the right of a query tile's diagonal are never loaded or
//     multiplied; only the diagonal tile applies an element mask.
//   * Epilogue: O / l -> fp16/bf16 -> swizzled shared memory -> TMA store; lse in fp32.
//
// Every wait is bounded (mbarrier try_wait against %globaltimer). On timeout the CTA records
// an error bit in `status`, all roles leave their loops, outstanding TMA loads and MMAs are
// drained, TMEM is freed and the kernel returns.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "ptx.cuh"

namespace fa {

constexpr int kBM = 128;        // query rows per query tile (tcgen05 M)
constexpr int kBN = 128;        // keys per K/V tile (tcgen05 N of S = QK^T)
constexpr int kQTiles = 2;      // query tiles per work item
constexpr int kItemRows = kBM * kQTiles;
constexpr int kNumThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kTmemCols = 512;  // S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D)
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

// Status bits written by the kernel (host reads them through fa_check_device_status).
constexpr unsigned kStatusTimeout = 1u;

struct Params {
  CUtensorMap tm_q;  // [BH, N, D] viewed as 3-D (D, N, BH), box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;  // same view, box (64, 32, 1): each softmax warp stores its own 32 rows
  float* lse;                  // [BH, N] fp32 or nullptr
  unsigned int* status;        // device word; error bits are OR-ed in
  unsigned long long timeout_ns;
  int BH;
  int N;
  int num_mb;                  // ceil(N / 256)
  int num_items;               // BH * num_mb
  int section;                 // causal ordering: heads per L2 section
  float scale_log2;            // scale * log2(e)
};

template <int D>
struct SmemLayout {
  static constexpr int kChunks = D / 64;           // 64-column (128-byte) swizzle chunks per row
  static constexpr int kChunkBytes = kBM * 128;    // one chunk of a 128-row tile
  static constexpr int kTileBytes = kBM * D * 2;   // a 128 x D fp16/bf16 tile
  static constexpr int kStages = (D == 64) ? 6 : 3;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kOOff = kKVOff + kStages * kTileBytes;
  static constexpr int kBarOff = kOOff + kQTiles * kTileBytes;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 1;
  static constexpr int kKVFull = 2;
  static constexpr int kKVEmpty = kKVFull + kStages;
  static constexpr int kSFull = kKVEmpty + kStages;  // [2]
  static constexpr int kPFull = kSFull + 2;          // [2]
  static constexpr int kOFull = kPFull + 2;          // [2]
  static constexpr int kDrain = kOFull + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynamicBytes = kBytes + 1024;  // slack to align the base to 1024 bytes
  static_assert(kDynamicBytes <= 232448, "shared memory budget");
};

struct Watch {
  volatile int* abort_flag;
  unsigned int* status;
  unsigned long long limit_ns;
};

// Bounded wait on an mbarrier phase. Returns false on timeout or when another role aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Watch& w, unsigned site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (global_timer_ns() - t0 > w.limit_ns) {
      *w.abort_flag = 1;
      atomicOr(w.status, kStatusTimeout | (1u << (8 + (site & 15))));
      return false;
    }
  }
}

// Wait used only while tearing down after an abort: ignores the abort flag, fixed limit.
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) return false;
  }
  return true;
}

struct Item {
  int bh;
  int mb;
};

// Work-item order. Non-causal: head-major (all row blocks of a head run close together, so
// the head's K/V is read from DRAM about once). Causal: heads are grouped into sections that
// fit in L2; inside a section the most expensive row blocks (largest mb) come first.
template <bool CAUSAL>
__device__ __forceinline__ Item decode_item(int t, const Params& p) {
  Item it;
  if (!CAUSAL) {
    it.bh = t / p.num_mb;
    it.mb = t - it.bh * p.num_mb;
  } else {
    const int per_sec = p.section * p.num_mb;
    const int sec = t / per_sec;
    const int r = t - sec * per_sec;
    const int hs = min(p.section, p.BH - sec * p.section);
    it.mb = p.num_mb - 1 - r / hs;
    it.bh = sec * p.section + (r - (r / hs) * hs);
  }
  return it;
}

// Number of K/V tiles each query tile of row block mb visits (0 = tile lies beyond N).
template <bool CAUSAL>
__device__ __forceinline__ void tile_counts(int mb, int N, int& n0, int& n1) {
  const int nkt = (N + kBN - 1) / kBN;
  const bool t1 = mb * kItemRows + kBM < N;
  if (CAUSAL) {
    n0 = min(2 * mb + 1, nkt);
    n1 = t1 ? min(2 * mb + 2, nkt) : 0;
  } else {
    n0 = nkt;
    n1 = t1 ? nkt : 0;
  }
}

// k-th work item of this CTA in snake order over the sorted item list (-1 when done).
__device__ __forceinline__ int item_of(int k, int num_items) {
  const int G = gridDim.x;
  const long long base = static_cast<long long>(k) * G;
  if (base >= num_items) return -1;
  const int c = (k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long t = base + c;
  return t < num_items ? static_cast<int>(t) : -1;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kNumThreads, 1) fa_fwd_kernel(const __grid_constant__ Params p) {
  using L = SmemLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](int idx) -> uint32_t { return sbase + L::kBarOff + 8u * idx; };
  auto q_addr = [&](int i) -> uint32_t { return sbase + L::kQOff + i * L::kTileBytes; };
  auto kv_addr = [&](int s) -> uint32_t { return sbase + L::kKVOff + s * L::kTileBytes; };
  auto o_addr = [&](int i) -> uint32_t { return sbase + L::kOOff + i * L::kTileBytes; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const Watch watch{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kKVFull + s), 1);
      mbar_init(bar(L::kKVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kSFull + i), 1);
      mbar_init(bar(L::kPFull + i), kBM);
      mbar_init(bar(L::kOFull + i), 1);
    }
    mbar_init(bar(L::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_o);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_pos = 0, q_loads = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int t = item_of(k, p.num_items);
        if (t < 0) break;
        const Item it = decode_item<CAUSAL>(t, p);
        int n0, n1;
        tile_counts<CAUSAL>(it.mb, p.N, n0, n1);
        const int nk = max(n0, n1);
        // Q tiles: wait until every S MMA of the previous item has read them.
        if (!(ok = wait_phase(bar(L::kQEmpty), (q_loads & 1) ^ 1, watch, 0))) break;
        const int nq = n1 > 0 ? 2 : 1;
        mbar_arrive_expect_tx(bar(L::kQFull), nq * L::kTileBytes);
        for (int i = 0; i < nq; ++i)
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(q_addr(i) + c * L::kChunkBytes, &p.tm_q, bar(L::kQFull), c * 64,
                        it.mb * kItemRows + i * kBM, it.bh);
        ++q_loads;
        for (int j = 0; j < nk && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t s = kv_pos % L::kStages;
            const uint32_t ph = (kv_pos / L::kStages) & 1;
            if (!(ok = wait_phase(bar(L::kKVEmpty + s), ph ^ 1, watch, 1))) break;
            mbar_arrive_expect_tx(bar(L::kKVFull + s), L::kTileBytes);
            const void* tm = kv == 0 ? static_cast<const void*>(&p.tm_k) : static_cast<const void*>(&p.tm_v);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(kv_addr(s) + c * L::kChunkBytes, tm, bar(L::kKVFull + s), c * 64, j * kBN, it.bh);
            ++kv_pos;
          }
        }
      }
      if (!ok) {
        // Let every load already issued land before the CTA can exit.
        if (q_loads > 0) wait_phase_drain(bar(L::kQFull), (q_loads - 1) & 1);
        for (uint32_t s = 0; s < static_cast<uint32_t>(L::kStages); ++s) {
          if (kv_pos <= s) continue;
          const uint32_t last = kv_pos - 1 - ((kv_pos - 1 - s) % L::kStages);
          wait_phase_drain(bar(L::kKVFull + s), (last / L::kStages) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc_f16(BF16, kBM, kBN, false);
      constexpr uint32_t idesc_o = instr_desc_f16(BF16, kBM, D, true);
      uint32_t kv_pos = 0, items = 0;
      uint32_t pcnt[2] = {0, 0};
      bool ok = true;

      // S_i = Q_i K^T into TMEM columns [128 i, 128 i + 128).
      auto issue_s = [&](int i, uint32_t stage) {
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(i * kBN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          const uint64_t a = smem_desc_sw128(q_addr(i) + off, 16, 1024);
          const uint64_t b = smem_desc_sw128(kv_addr(stage) + off, 16, 1024);
          mma_ss(d_tmem, a, b, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      // O_i (+)= P_i V; P_i (fp16/bf16, 64 columns) sits in the first half of S_i's columns.
      auto issue_pv = [&](int i, uint32_t stage, bool accumulate) {
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(2 * kBN + i * D);
        const uint32_t a_tmem = tmem + static_cast<uint32_t>(i * kBN);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // V tile: keys are the K dimension (rows, 128 B apart), D is the N dimension
          // (MN-major): 8-key groups are 1024 B apart, 64-column chunks kChunkBytes apart.
          const uint64_t b = smem_desc_sw128(kv_addr(stage) + kk * 16 * 128, L::kChunkBytes, 1024);
          mma_ts(d_tmem, a_tmem + kk * 8, b, idesc_o, (accumulate || kk > 0) ? 1u : 0u);
        }
      };

      for (int k = 0; ok; ++k) {
        const int t = item_of(k, p.num_items);
        if (t < 0) break;
        const Item it = decode_item<CAUSAL>(t, p);
        int n[2];
        tile_counts<CAUSAL>(it.mb, p.N, n[0], n[1]);
        const int nk = max(n[0], n[1]);
        if (!(ok = wait_phase(bar(L::kQFull), items & 1, watch, 2))) break;
        // prologue: S_i for K tile 0
        uint32_t sk = kv_pos % L::kStages;
        if (!(ok = wait_phase(bar(L::kKVFull + sk), (kv_pos / L::kStages) & 1, watch, 3))) break;
        ++kv_pos;
        tc_fence_after();
        for (int i = 0; i < 2; ++i)
          if (n[i] > 0) {
            issue_s(i, sk);
            mma_commit(bar(L::kSFull + i));
          }
        mma_commit(bar(L::kKVEmpty + sk));
        for (int j = 0; j < nk && ok; ++j) {
          const uint32_t sv = kv_pos % L::kStages;
          if (!(ok = wait_phase(bar(L::kKVFull + sv), (kv_pos / L::kStages) & 1, watch, 4))) break;
          ++kv_pos;
          tc_fence_after();
          bool k_next = false;
          uint32_t sk2 = 0;
          for (int i = 0; i < 2 && ok; ++i) {
            if (j < n[i]) {
              if (!(ok = wait_phase(bar(L::kPFull + i), pcnt[i] & 1, watch, 5 + i))) break;
              ++pcnt[i];
              tc_fence_after();
              issue_pv(i, sv, j > 0);
              if (j == n[i] - 1) mma_commit(bar(L::kOFull + i));
            }
            if (j + 1 < n[i]) {
              if (!k_next) {
                sk2 = kv_pos % L::kStages;
                if (!(ok = wait_phase(bar(L::kKVFull + sk2), (kv_pos / L::kStages) & 1, watch, 7))) break;
                ++kv_pos;
                tc_fence_after();
                k_next = true;
              }
              issue_s(i, sk2);
              mma_commit(bar(L::kSFull + i));
            }
          }
          if (!ok) break;
          mma_commit(bar(L::kKVEmpty + sv));
          if (k_next) mma_commit(bar(L::kKVEmpty + sk2));
        }
        if (!ok) break;
        mma_commit(bar(L::kQEmpty));
        ++items;
      }
      // Whatever happened, wait for every issued MMA before TMEM can be freed.
      mma_commit(bar(L::kDrain));
      wait_phase_drain(bar(L::kDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;        // query tile of the item handled by this warpgroup
    const int wq = warp & 3;         // TMEM lane quarter accessible to this warp
    const int r = wq * 32 + lane;    // row within the query tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + static_cast<uint32_t>(wg * kBN);
    const uint32_t t_o = tmem + lane_off + static_cast<uint32_t>(2 * kBN + wg * D);
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, ocnt = 0;
    bool ok = true;

    for (int k = 0; ok; ++k) {
      const int t = item_of(k, p.num_items);
      if (t < 0) break;
      const Item it = decode_item<CAUSAL>(t, p);
      int n0, n1;
      tile_counts<CAUSAL>(it.mb, p.N, n0, n1);
      const int n_mine = wg == 0 ? n0 : n1;
      if (n_mine == 0) continue;
      const int row = it.mb * kItemRows + wg * kBM + r;  // query index within the sequence
      const int qt = 2 * it.mb + wg;                     // query tile index (diagonal K tile)
      float m_used = -INFINITY;
      float l_run = 0.f;

      for (int j = 0; j < n_mine; ++j) {
        bool w_ok = wait_phase(bar(L::kSFull + wg), scnt & 1, watch, 8 + wg);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        ++scnt;
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld32x32b_x128(t_s, sr);
        float* s = reinterpret_cast<float*>(sr);

        const int col0 = j * kBN;
        const bool diag = CAUSAL && j == qt;
        if (diag || col0 + kBN > p.N) {
          int lim = p.N - 1 - col0;
          if (diag) lim = min(lim, row - col0);
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < kBN; c += 4) {
          mx0 = fmaxf(mx0, s[c]);
          mx1 = fmaxf(mx1, s[c + 1]);
          mx2 = fmaxf(mx2, s[c + 2]);
          mx3 = fmaxf(mx3, s[c + 3]);
        }
        const float x_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_used = x_max;
        } else if (x_max > m_used + kRescaleLog2) {
          alpha = ex2_approx(m_used - x_max);
          m_used = x_max;
          l_run *= alpha;
          rescale = true;
        }
        const float neg_m = -m_used;
        float ls0 = 0.f, ls1 = 0.f;
        uint32_t pk[kBN / 2];
#pragma unroll
        for (int c = 0; c < kBN / 2; ++c) {
          const float p0 = ex2_approx(fmaf(s[2 * c], sl2, neg_m));
          const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl2, neg_m));
          ls0 += p0;
          ls1 += p1;
          pk[c] = pack2<BF16>(p0, p1);
        }
        l_run += ls0 + ls1;
        tmem_st32x32b_x64(t_s, pk);
        if (__any_sync(0xffffffffu, rescale)) {
          // O row *= alpha (alpha = 1 for rows that keep their max). The PV MMA of the
          // previous tile has completed: S of this tile was issued after it.
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32x32b_x32(t_o + c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32x32b_x32(t_o + c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::kPFull + wg));
      }
      if (!ok) break;

      // ---------------- epilogue: O / l -> staging shared memory -> TMA store; lse
      // Each warp stages and stores its own 32 rows, so no barrier spans warps.
      bool e_ok = wait_phase(bar(L::kOFull + wg), ocnt & 1, watch, 10 + wg);
      ++ocnt;
      if (!__all_sync(0xffffffffu, e_ok)) {
        ok = false;
        break;
      }
      if (lane == 0) bulk_wait_group_read0();  // this warp's previous store has left the buffer
      __syncwarp();
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const uint32_t ob = o_addr(wg);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32x32b_x32(t_o + c, o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = c + 8 * u;         // first of the 8 columns in this 16-byte unit
          const int chunk = col >> 6;        // 64-column swizzle chunk
          const int unit = (col & 63) >> 3;  // 16-byte unit within the 128-byte row
          const uint32_t addr = ob + chunk * L::kChunkBytes + r * 128 + ((unit ^ (r & 7)) << 4);
          const uint32_t w0 = pack2<BF16>(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l);
          const uint32_t w1 = pack2<BF16>(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l);
          const uint32_t w2 = pack2<BF16>(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l);
          const uint32_t w3 = pack2<BF16>(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
      }
      if (p.lse != nullptr && row < p.N)
        p.lse[static_cast<long long>(it.bh) * p.N + row] = (m_used + log2f(l_run)) * kLn2;
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      const int row0_warp = it.mb * kItemRows + wg * kBM + wq * 32;
      if (lane == 0 && row0_warp < p.N) {  // rows past N are clipped by the store; skip empty boxes
        for (int c = 0; c < L::kChunks; ++c)
          tma_store_3d(&p.tm_o, ob + c * L::kChunkBytes + wq * 32 * 128, c * 64, row0_warp, it.bh);
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
