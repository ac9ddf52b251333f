// fp32-I/O attention forward for sm_103a: Q, K, V, O stored in fp32, the two matmuls on the
// tensor cores in tf32 (tcgen05.mma kind::tf32, fp32 accumulation), softmax in fp32.
//
// This is the pages' second storage variant: "Android Transformer Optimization: Attention and
// Mobile GPU Bottlenecks" (section "Pitfalls I Hit") keeps an fp32-storage build beside the
// fp16 one, with the tile cut in half because each element takes twice the bytes. Here the
// key tiles are 64 keys (half of the 16-bit kernel's 128) so that a K or V tile takes the
// same shared memory as there; query tiles stay 128 rows (the tcgen05 M).
//
// Structure (one CTA per SM, 384 threads), the single-query-tile form of the 16-bit kernel:
//   warps 0-3, 4-7  softmax warpgroups: warpgroup w takes the key tiles j with j % 2 == w of
//                   the item's query tile; warpgroup 0 merges both partial (m, l, O) at the end
//   warp 8          MMA issuer (whole warp, one elected lane issues) and TMEM owner
//   warp 9          TMA producer
//   warps 10-11     V transposers: copy each V tile, in 4 x 4 blocks, into a K-major tile (Vt)
//                   for the PV product (the MMAs here read tf32 operands K-major)
// K and V tiles stream through separate rings: the MMA warp is the only reader of the K ring
// and the transposers the only readers of the V ring, so each waits on every position of its
// ring in order and an mbarrier phase can never be mistaken for one two phases later.
// TMEM: S_w (fp32, 64 columns) at 64 w; P_w (tf32, rounded to nearest) overwrites S_w; O_w
// (fp32, D columns) at 128 + D w; Q (D columns) after them. Per warpgroup the MMA order is
// S(j), PV(j), S(j + 2), so the in-order tensor pipe keeps S(j + 2) from overwriting P(j)
// before PV(j) has read it.
//
// Q is copied from its TMA tile into TMEM once per item (tcgen05.cp) and S = Q K^T reads it
// there. With both operands in shared memory an S step reads 6 KB for 32 cycles of tensor
// work; steps that read 6 KB from shared memory were measured at 48 cycles (128 bytes per
// cycle). From TMEM only the 2 KB of K is read.
//
// Operand layouts (128-byte swizzle, 32 fp32 per 128-byte row segment):
//   Q tile  128 x D, as loaded by TMA; D / 32 chunks of 128 rows x 128 bytes, copied to TMEM
//   K tile  64 x D,  K-major B of S;           D / 32 chunks of 64 rows x 128 bytes
//   V tile  64 x D,  as loaded (keys are rows); transposed in shared memory into
//   Vt      D x 64,  K-major B of O += P V (D is N, keys are K); 2 chunks of D rows x 128 bytes
// A tf32 MMA step covers K = 8 (32 bytes of a row segment), like the 16-element step of f16.
#pragma once

#include "fa_kernel.cuh"

namespace fa {

constexpr int kBNf = 64;  // keys per K/V tile in the fp32 kernel

template <int D>
struct SmemLayoutF32 {
  static constexpr int kChunks = D / 32;               // 128-byte (32 x fp32) chunks per row
  static constexpr int kQChunkBytes = kBM * 128;       // one chunk of the 128-row Q tile
  static constexpr int kKVChunkBytes = kBNf * 128;     // one chunk of a 64-row K or V tile
  static constexpr int kQBytes = kBM * D * 4;
  static constexpr int kKVBytes = kBNf * D * 4;
  static constexpr int kKStages = (D == 64) ? 4 : 2;          // K ring
  static constexpr int kVStages = (D == 64) ? 2 : 1;          // V ring
  static constexpr int kNumVt = (D == 64) ? 2 : 1;            // transposed V buffers
  static constexpr int kVtChunkBytes = D * 128;              // 32 keys of all D rows
  static constexpr int kOCols = 64;                           // O columns staged per pass
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kKStages * kKVBytes;
  static constexpr int kVtOff = kVOff + kVStages * kKVBytes;
  static constexpr int kOOff = kVtOff + kNumVt * kKVBytes;   // O staging of warpgroup 0
  static constexpr int kOWarpBytes = 32 * kOCols * 4;        // one warp's 32 rows x kOCols fp32
  static constexpr int kOBytes = 4 * kOWarpBytes;
  static constexpr int kStatsOff = kOOff + kOBytes;          // (m, l) hand-off, 2 x 128 fp32
  static constexpr int kBarOff = kStatsOff + 2 * kBM * 4;
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 1;
  static constexpr int kKFull = 2;
  static constexpr int kKEmpty = kKFull + kKStages;
  static constexpr int kVFull = kKEmpty + kKStages;
  static constexpr int kVEmpty = kVFull + kVStages;  // 64 transposer arrivals
  static constexpr int kSFull = kVEmpty + kVStages;  // [2]
  static constexpr int kPFull = kSFull + 2;          // [2]
  static constexpr int kOFull = kPFull + 2;          // [2]
  static constexpr int kVtFull = kOFull + 2;        // [kNumVt] 64 transposer arrivals
  static constexpr int kVtEmpty = kVtFull + kNumVt;  // [kNumVt] the PV that read it completed
  static constexpr int kStats = kVtEmpty + kNumVt;
  static constexpr int kO1Free = kStats + 1;
  static constexpr int kDrain = kO1Free + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynamicBytes = kBytes + 1024;
  static_assert(kDynamicBytes <= 232448, "shared memory budget");
  // TMEM: S_w (64 columns) at 64 w, O_w (D columns) at 128 + D w, Q (tf32, D columns) after them.
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kQCol = 2 * kBNf + 2 * D;
  static_assert(kQCol + D <= kTmemCols, "TMEM budget");
};

// tcgen05 instruction descriptor, kind::tf32: D fp32, A and B tf32 (format 2).
__host__ __device__ constexpr uint32_t instr_desc_tf32(int M, int N, bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Copies a 128-row x 256-bit slice of a shared-memory matrix (the layout its descriptor gives)
// into 128 TMEM lanes x 8 columns; asynchronous, ordered before later tcgen05.mma of this thread.
__device__ __forceinline__ void tmem_cp_128x256b_leader(uint32_t taddr, uint64_t s_desc, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %2, 0;\n\t"
      "@q tcgen05.cp.cta_group::1.128x256b [%0], %1;\n\t}" ::"r"(taddr),
      "l"(s_desc), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_ts_tf32_leader(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
// fp32 -> tf32, rounded to nearest (ties away from zero), in a 32-bit register: half a tf32
// unit (bit 12) is added to the fp32 bits, and the tensor core, which reads the top 19 bits of
// a tf32 operand, drops the rest. For finite x >= 0 (every P) this gives the bits of
// cvt.rna.tf32.f32 in one integer add; the kernel's outputs were measured bit-identical.
__device__ __forceinline__ uint32_t to_tf32_for_mma(float x) { return __float_as_uint(x) + 0x1000u; }

// Key tiles (64 keys) of the item's query tile: all of them, or causally those that hold a
// key <= the tile's last row; warpgroup w processes tiles j = w, w + 2, ...
template <bool CAUSAL>
__host__ __device__ inline void tile_counts_f32(int qt, int N, int& nk, int& n0, int& n1) {
  const int nkt = (N + kBNf - 1) / kBNf;
  nk = CAUSAL ? min(2 * qt + 2, nkt) : nkt;
  n0 = (nk + 1) >> 1;
  n1 = nk >> 1;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kNumThreads, 1) fa_fwd_f32_kernel(const __grid_constant__ Params p) {
  using L = SmemLayoutF32<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](int idx) -> uint32_t { return sbase + L::kBarOff + 8u * idx; };
  const uint32_t q_base = sbase + L::kQOff;
  auto k_addr = [&](int s) -> uint32_t { return sbase + L::kKOff + s * L::kKVBytes; };
  auto v_addr = [&](int s) -> uint32_t { return sbase + L::kVOff + s * L::kKVBytes; };
  auto vt_addr = [&](int b) -> uint32_t { return sbase + L::kVtOff + b * L::kKVBytes; };
  float* stats_m = reinterpret_cast<float*>(smem + L::kStatsOff);
  float* stats_l = stats_m + kBM;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const Watch watch{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), 1);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 64);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kSFull + i), 1);
      mbar_init(bar(L::kPFull + i), kBM);
      mbar_init(bar(L::kOFull + i), 1);
    }
    for (int i = 0; i < L::kNumVt; ++i) {
      mbar_init(bar(L::kVtFull + i), 64);
      mbar_init(bar(L::kVtEmpty + i), 1);
    }
    mbar_init(bar(L::kStats), kBM);
    mbar_init(bar(L::kO1Free), kBM);
    mbar_init(bar(L::kDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // The producer decodes its first item during setup (parameters and work table only), off the
  // path to the first Q load.
  const int t_first = (warp == kLoadWarp && lane == 0) ? item_of(0, p) : -1;
  Item it_first{};
  int nk_first = 0, n0_first = 0, n1_first = 0;
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_o);
    if (t_first >= 0) {
      it_first = decode_item<CAUSAL>(t_first, p);
      tile_counts_f32<CAUSAL>(it_first.mb, p.N, nk_first, n0_first, n1_first);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  grid_dependency_wait();

  if (warp >= 8) {
    if (warp == kLoadWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        uint32_t k_pos = 0, v_pos = 0, q_loads = 0;
        bool ok = true;
        // One tile into the K ring (is_v = false) or the V ring, at that ring's next position.
        auto load_tile = [&](bool is_v, int j, int bh) -> bool {
          uint32_t& pos = is_v ? v_pos : k_pos;
          const int nst = is_v ? L::kVStages : L::kKStages;
          const uint32_t s = pos % nst;
          const uint32_t full = bar((is_v ? L::kVFull : L::kKFull) + s);
          if (!wait_phase(bar((is_v ? L::kVEmpty : L::kKEmpty) + s), ((pos / nst) & 1) ^ 1, watch, 1)) return false;
          mbar_arrive_expect_tx(full, L::kKVBytes);
          const uint32_t dst = is_v ? v_addr(s) : k_addr(s);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(dst + c * L::kKVChunkBytes, is_v ? &p.tm_v : &p.tm_k, full, c * 32, j * kBNf, bh);
          ++pos;
          return true;
        };
        for (int k = 0; ok; ++k) {
          const int t = k == 0 ? t_first : item_of(k, p);
          if (t < 0) break;
          const Item it = k == 0 ? it_first : decode_item<CAUSAL>(t, p);
          int nk = nk_first, n0 = n0_first, n1 = n1_first;
          if (k > 0) tile_counts_f32<CAUSAL>(it.mb, p.N, nk, n0, n1);
          if (!(ok = wait_phase(bar(L::kQEmpty), (q_loads & 1) ^ 1, watch, 0))) break;
          mbar_arrive_expect_tx(bar(L::kQFull), L::kQBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(q_base + c * L::kQChunkBytes, &p.tm_q, bar(L::kQFull), c * 32, it.mb * kBM, it.bh);
          ++q_loads;
          // In the order they are needed: K0 K1 V0 K2 V1 K3 V2 ...
          ok = load_tile(false, 0, it.bh);
          for (int j = 0; j < nk && ok; ++j) {
            if (j + 1 < nk) ok = load_tile(false, j + 1, it.bh);
            ok = ok && load_tile(true, j, it.bh);
          }
        }
        if (!ok) {
          // Let every load already issued land before the CTA can exit.
          if (q_loads > 0) wait_phase_drain(bar(L::kQFull), (q_loads - 1) & 1);
          for (int ring = 0; ring < 2; ++ring) {
            const uint32_t pos = ring ? v_pos : k_pos;
            const uint32_t nst = ring ? L::kVStages : L::kKStages;
            for (uint32_t s = 0; s < nst; ++s) {
              if (pos <= s) continue;
              const uint32_t last = pos - 1 - ((pos - 1 - s) % nst);
              wait_phase_drain(bar((ring ? L::kVFull : L::kKFull) + s), (last / nst) & 1);
            }
          }
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t leader = elect_one_lane();
      constexpr uint32_t idesc_s = instr_desc_tf32(kBM, kBNf, false);
      constexpr uint32_t idesc_o = instr_desc_tf32(kBM, D, false);
      uint32_t k_pos = 0, items = 0, merges = 0, pcnt0 = 0, pcnt1 = 0;
      bool ok = true;
      auto wait = [&](uint32_t b, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, wait_phase(b, parity, watch, site));
      };
      auto next_k = [&](uint32_t& stage) -> bool {
        stage = k_pos % L::kKStages;
        if (!wait(bar(L::kKFull + stage), (k_pos / L::kKStages) & 1, 3)) return false;
        ++k_pos;
        tc_fence_after();
        return true;
      };
      const uint64_t q_desc = smem_desc_sw128(q_base, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(k_addr(0), 16, 1024);
      const uint64_t vt_desc = smem_desc_sw128(vt_addr(0), 16, 1024);
      constexpr uint32_t kStageEnc = L::kKVBytes >> 4;
      uint32_t vt_cnt = 0;  // V tiles consumed (transposed buffers used in turn)
      // S_w = Q K^T (64 columns at 64 w): D / 8 steps of K = 8. A is Q in TMEM (8 columns per
      // step), B the K tile in shared memory (32 bytes of a row segment per step).
      auto issue_s = [&](int w, uint32_t stage) {
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(w * kBNf);
        const uint64_t b0 = k_desc + stage * kStageEnc;
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk) {
          const uint32_t b_off = ((kk >> 2) * L::kKVChunkBytes + (kk & 3) * 32) >> 4;
          mma_ts_tf32_leader(d_tmem, tmem + L::kQCol + 8 * kk, b0 + b_off, idesc_s, kk > 0 ? 1u : 0u, leader);
        }
        mma_commit_leader(bar(L::kSFull + w), leader);
      };
      // The next transposed V tile (written by the transposers, in V order).
      auto next_vt = [&](uint32_t& buf) -> bool {
        buf = vt_cnt % L::kNumVt;
        if (!wait(bar(L::kVtFull + buf), (vt_cnt / L::kNumVt) & 1, 4)) return false;
        ++vt_cnt;
        tc_fence_after();
        return true;
      };
      // O_w (+)= P_w V: P_w is tf32 in S_w's 64 columns; B = Vt, K-major (D rows, the keys in
      // two 128-byte chunks kVtChunkBytes apart; a step of 8 keys is 32 bytes of a row segment).
      auto issue_pv = [&](int w, uint32_t buf, bool accumulate, bool last) -> bool {
        const uint32_t pc = w ? pcnt1 : pcnt0;
        if (!wait(bar(L::kPFull + w), pc & 1, 5 + w)) return false;
        if (w) ++pcnt1;
        else ++pcnt0;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(2 * kBNf + w * D);
        const uint32_t a_tmem = tmem + static_cast<uint32_t>(w * kBNf);
        const uint64_t b0 = vt_desc + buf * kStageEnc;
#pragma unroll
        for (int kk = 0; kk < kBNf / 8; ++kk)
          mma_ts_tf32_leader(d_tmem, a_tmem + kk * 8, b0 + (((kk >> 2) * L::kVtChunkBytes + (kk & 3) * 32) >> 4),
                             idesc_o, (accumulate || kk > 0) ? 1u : 0u, leader);
        mma_commit_leader(bar(L::kVtEmpty + buf), leader);
        if (last) mma_commit_leader(bar(L::kOFull + w), leader);
        return true;
      };
      auto release = [&](uint32_t stage) { mma_commit_leader(bar(L::kKEmpty + stage), leader); };

      for (int k = 0; ok; ++k) {
        const int t = item_of(k, p);
        if (t < 0) break;
        const Item it = decode_item<CAUSAL>(t, p);
        int nk, n0, n1;
        tile_counts_f32<CAUSAL>(it.mb, p.N, nk, n0, n1);
        if (!(ok = wait(bar(L::kQFull), items & 1, 2))) break;
        tc_fence_after();
        // Q into TMEM, one 8-column step of K at a time. The copies follow the previous item's
        // last S MMA in issue order, and the shared-memory Q tile is free for the next item's
        // load once they complete.
#pragma unroll
        for (int kk = 0; kk < D / 8; ++kk)
          tmem_cp_128x256b_leader(tmem + L::kQCol + 8 * kk,
                                  q_desc + (((kk >> 2) * L::kQChunkBytes + (kk & 3) * 32) >> 4), leader);
        mma_commit_leader(bar(L::kQEmpty), leader);
        uint32_t sk, sv;
        // S_0(K0), S_1(K1), then per j: PV_{j&1}(V_j), S_{j&1}(K_{j+2}).
        if (!(ok = next_k(sk))) break;
        issue_s(0, sk);
        release(sk);
        if (nk > 1) {
          if (!(ok = next_k(sk))) break;
          issue_s(1, sk);
          release(sk);
        }
        for (int j = 0; j < nk && ok; ++j) {
          const int w = j & 1;
          if (!(ok = next_vt(sv))) break;
          // O1 is overwritten by the first PV of warpgroup 1: the previous merge must have read it.
          if (j == 1 && merges > 0 && !(ok = wait(bar(L::kO1Free), (merges - 1) & 1, 13))) break;
          if (!(ok = issue_pv(w, sv, j >= 2, j + 2 >= nk))) break;
          if (j + 2 < nk) {
            if (!(ok = next_k(sk))) break;
            issue_s(w, sk);
            release(sk);
          }
        }
        if (ok && n1 > 0) ++merges;
        if (!ok) break;
        ++items;
      }
      mma_commit_leader(bar(L::kDrain), leader);
      if (leader) wait_phase_drain(bar(L::kDrain), 0);
      __syncwarp();
    } else {
      // ------------------------------------------------------------ V transposers (warps 10-11)
      // Element (key, d) of a V tile (64 keys x D fp32 as loaded: 128-byte swizzled chunks of
      // 32 columns) goes to row d of Vt (K-major: the 64 keys of a row in two 128-byte swizzled
      // chunks). V ring positions and transposed buffers are both taken in V order.
      const int t = threadIdx.x - 320;  // 0..63
      uint32_t v_pos = 0, vt_cnt = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int ti = item_of(k, p);
        if (ti < 0) break;
        const Item it = decode_item<CAUSAL>(ti, p);
        int nk, n0, n1;
        tile_counts_f32<CAUSAL>(it.mb, p.N, nk, n0, n1);
        for (int j = 0; j < nk && ok; ++j) {
          const uint32_t stage = v_pos % L::kVStages;
          const uint32_t buf = vt_cnt % L::kNumVt;
          if (!(ok = wait_phase(bar(L::kVFull + stage), (v_pos / L::kVStages) & 1, watch, 15))) break;
          if (!(ok = wait_phase(bar(L::kVtEmpty + buf), ((vt_cnt / L::kNumVt) & 1) ^ 1, watch, 15))) break;
          ++v_pos;
          ++vt_cnt;
          // 4 x 4 blocks (keys 4g .. 4g + 3, columns 4uf .. 4uf + 3): four 16-byte loads of V
          // rows, four 16-byte stores of Vt rows. The eight lanes of a quarter warp take one
          // diagonal of an 8 x 8 grid of blocks, so each load and each store touches eight
          // distinct 16-byte bank groups.
          {
            constexpr int kColChunks = D / 32;
            constexpr int kPerQuarter = 2 * kColChunks;  // (2 key chunks x kColChunks x 8 diagonals) / 8 quarters
            const int quarter = t >> 3, l8 = t & 7;
            const uint32_t vsrc = v_addr(stage), vdst = vt_addr(buf);
#pragma unroll 2
            for (int k2 = 0; k2 < kPerQuarter; ++k2) {
              const int idx = quarter * kPerQuarter + k2;
              const int sft = idx & 7, C = (idx >> 3) % kColChunks, G = idx / (8 * kColChunks);
              const int g = 8 * G + l8;
              const int u = (l8 + sft) & 7;
              const int uf = 8 * C + u;
              uint32_t x[4][4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int r = 4 * g + i;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(x[i][0]), "=r"(x[i][1]), "=r"(x[i][2]), "=r"(x[i][3])
                             : "r"(vsrc + C * L::kKVChunkBytes + r * 128 + ((u ^ (r & 7)) << 4)));
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int d = 4 * uf + e;
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(vdst + G * L::kVtChunkBytes + d * 128 +
                                                                            (((g & 7) ^ (d & 7)) << 4)),
                             "r"(x[0][e]), "r"(x[1][e]), "r"(x[2][e]), "r"(x[3][e])
                             : "memory");
              }
            }
          }
          fence_proxy_async_smem();  // the MMA (async proxy) reads Vt; TMA refills the V stage
          mbar_arrive(bar(L::kVEmpty + stage));
          mbar_arrive(bar(L::kVtFull + buf));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + static_cast<uint32_t>(wg * kBNf);
    const uint32_t t_o = tmem + lane_off + static_cast<uint32_t>(2 * kBNf + wg * D);
    const uint32_t t_o1 = tmem + lane_off + static_cast<uint32_t>(2 * kBNf + D);
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, ocnt = 0, o1cnt = 0, mcnt = 0;
    bool ok = true;

    for (int k = 0; ok; ++k) {
      const int t = item_of(k, p);
      if (t < 0) break;
      const Item it = decode_item<CAUSAL>(t, p);
      int nk, n0, n1;
      tile_counts_f32<CAUSAL>(it.mb, p.N, nk, n0, n1);
      const int n_mine = wg == 0 ? n0 : n1;
      if (n_mine == 0) continue;
      const int qt = it.mb;
      const int row = qt * kBM + r;
      float m_used = -INFINITY;  // may stay -inf: a causal key tile can hide every key of a row
      float l_run = 0.f;

      for (int jj = 0; jj < n_mine; ++jj) {
        const int j = 2 * jj + wg;
        const bool w_ok = wait_phase(bar(L::kSFull + wg), scnt & 1, watch, 8 + wg);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        ++scnt;
        tc_fence_after();
        uint32_t sr[kBNf];
        tmem_ld32x32b_x64(t_s, sr);
        float* s = reinterpret_cast<float*>(sr);
        const int col0 = j * kBNf;
        int lim = p.N - 1 - col0;
        if (CAUSAL) lim = min(lim, row - col0);
        if (lim < kBNf - 1) {
#pragma unroll
          for (int c = 0; c < kBNf; ++c)
            if (c > lim) s[c] = -INFINITY;
        }
        float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int c = 4; c < kBNf; c += 4)
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], s[c + i]);
        const float x_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
        float alpha = 1.f;
        bool rescale = false;
        if (jj == 0) {
          m_used = x_max;
        } else if (x_max > m_used + kRescaleLog2) {
          alpha = ex2_approx(m_used - x_max);  // 0 when m_used is still -inf
          m_used = x_max;
          l_run *= alpha;
          rescale = true;
        }
        const float m_base = m_used == -INFINITY ? 0.f : m_used;  // every key of this row masked so far
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kBNf; ++c) {
          const float pv = ex2_approx(fmaf(s[c], sl2, -m_base));
          acc[c & 3] += pv;
          sr[c] = to_tf32_for_mma(pv);
        }
        l_run += (acc[0] + acc[1]) + (acc[2] + acc[3]);
        tmem_st32x32b_x64(t_s, sr);  // P over S
        if (__any_sync(0xffffffffu, rescale)) {
          // O *= alpha. PV(j - 2) of this warpgroup is complete: it was issued before S(j).
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

      if (wg == 1) {
        // Hand (m, l) of the odd key tiles to warpgroup 0 (after it has read the previous ones).
        if (mcnt > 0) {
          const bool f_ok = wait_phase(bar(L::kO1Free), (mcnt - 1) & 1, watch, 14);
          if (!__all_sync(0xffffffffu, f_ok)) {
            ok = false;
            break;
          }
        }
        ++mcnt;
        stats_m[r] = m_used;
        stats_l[r] = l_run;
        mbar_arrive(bar(L::kStats));
        continue;
      }

      // ---------------- epilogue (warpgroup 0): merge, O / l -> fp32 staging -> TMA store; lse
      bool e_ok = wait_phase(bar(L::kOFull + 0), ocnt & 1, watch, 10);
      ++ocnt;
      const bool merge = n1 > 0;
      float a_self = 1.f, a_other = 0.f;
      if (merge) {
        e_ok = e_ok && wait_phase(bar(L::kOFull + 1), o1cnt & 1, watch, 11);
        e_ok = e_ok && wait_phase(bar(L::kStats), mcnt & 1, watch, 12);
        ++o1cnt;
        ++mcnt;
      }
      if (!__all_sync(0xffffffffu, e_ok)) {
        ok = false;
        break;
      }
      if (merge) {
        const float m1 = stats_m[r], l1 = stats_l[r];
        const float m = fmaxf(m_used, m1);
        a_self = ex2_approx(m_used - m);
        a_other = ex2_approx(m1 - m);  // 0 when warpgroup 1 saw no key of this row
        l_run = l_run * a_self + l1 * a_other;
        m_used = m;
      }
      const float inv_l = 1.0f / l_run;
      const float c_self = a_self * inv_l, c_other = a_other * inv_l;
      // This warp's 32 rows, kOCols columns per pass: kOCols / 32 boxes of 32 rows x 32 fp32
      // (128-byte swizzled rows, 4 KB each), stored by TMA before the next pass reuses them.
      const uint32_t ob = sbase + L::kOOff + wq * L::kOWarpBytes;
      const int row0_warp = qt * kBM + wq * 32;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += L::kOCols) {
        if (lane == 0) bulk_wait_group_read0();  // the previous store has left the buffer
        __syncwarp();
        tc_fence_after();
#pragma unroll 1
        for (int c = c0; c < c0 + L::kOCols; c += 32) {
          uint32_t o[32];
          if (merge) {
            uint32_t o1[32];
            tmem_ld32x32b_x32_pair(t_o + c, t_o1 + c, o, o1);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * c_self + __uint_as_float(o1[e]) * c_other);
          } else {
            tmem_ld32x32b_x32(t_o + c, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * c_self);
          }
          const uint32_t box = ob + ((c - c0) >> 5) * 4096 + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + ((u ^ (lane & 7)) << 4)),
                         "r"(o[4 * u + 0]), "r"(o[4 * u + 1]), "r"(o[4 * u + 2]), "r"(o[4 * u + 3])
                         : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0_warp < p.N) {
          for (int b = 0; b < L::kOCols / 32; ++b)
            tma_store_3d(&p.tm_o, ob + b * 4096, c0 + b * 32, row0_warp, it.bh);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      if (merge) mbar_arrive(bar(L::kO1Free));  // O1 and (m1, l1) consumed
      if (p.lse != nullptr && row < p.N)
        p.lse[static_cast<long long>(it.bh) * p.N + row] = (m_used + log2f(l_run)) * kLn2;
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) grid_launch_dependents();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace fa
