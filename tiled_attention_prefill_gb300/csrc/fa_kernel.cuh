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
//   * One CTA per SM, 384 threads = 3 warpgroups:
//       warps 0-3   softmax warpgroup 0 (one thread per query row, TMEM lane = row)
//       warps 4-7   softmax warpgroup 1
//       warp  8     tcgen05 MMA issuer (warp-uniform, one elected lane issues) and TMEM owner;
//                   at D = 64 with two query tiles per item it issues for warpgroup 0 only
//       warp  9     TMA producer (one thread; during setup it also initialises the barriers
//                   and issues the first work unit's Q load)
//       warp 10     at D = 64 with two query tiles per item: MMA issuer for warpgroup 1
//       warps 10-11 otherwise idle
//     At D = 128, setmaxnreg moves registers from the third warpgroup (88 each) to the softmax
//     warpgroups (208 each); 88 + 2 * 208 = 3 * 168, the launch allocation. At D = 64 every
//     role fits in the launch allocation and no split is made.
//   * K and V tiles (128 keys x D) stream through a shared-memory ring filled by TMA
//     (128-byte swizzle) in exactly the order the MMA warp consumes them. Single-query-tile
//     items leave the second Q tile free, and the ring starts there, one stage deeper; at
//     D = 128 two-query-tile items stage O one 64-column chunk at a time for a fourth stage.
//   * S = Q K^T for a warpgroup goes to its own 128 TMEM columns (fp32). The warpgroup reads
//     its row of S (tcgen05.ld), writes P as fp16/bf16 into TMEM (at D = 128 over S's columns;
//     at D = 64 into 64 columns of its own, so that the next S can be computed while the
//     softmax runs), and the MMA warp computes O += P V with P read from TMEM. O (fp32, D
//     columns per warpgroup) stays in TMEM for the whole K/V loop.
//   * Two work decompositions (template SPLITK):
//       false: a work item is 256 query rows = two 128-row query tiles, one per warpgroup,
//              sharing every K/V tile loaded (half the K/V traffic per query row).
//       true:  a work item is one 128-row query tile; warpgroup 0 takes the even K/V tiles,
//              warpgroup 1 the odd ones, and warpgroup 0 merges the two partial (m, l, O) at
//              the end with the same rescaling rule. Twice the work items and half the serial
//              chain per item: used when there are too few items to fill the GPU.
//   * The max used in the exponent only moves when a tile raises the row max by more than
//     2^8; otherwise p = 2^(x - m_used) may exceed 1 (at most 256). O and l always carry the
//     same factor, so O / l is unchanged, and the O rescale in TMEM is rarely needed.
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
constexpr int kNumThreads = 384;
constexpr int kLaunchRegs = 168;   // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int kSoftmaxRegs = 208;  // after setmaxnreg, softmax warpgroups
constexpr int kOtherRegs = 88;     // after setmaxnreg, MMA / TMA / idle warpgroup
static_assert(kOtherRegs + 2 * kSoftmaxRegs <= 3 * kLaunchRegs, "register split exceeds the launch pool");
// The split is used at D = 128 only: at D = 64 every role fits the launch allocation without
// spilling, and the smaller MMA / TMA region would spill (measured 3-4% slower).
template <int D>
constexpr bool reg_split() { return D == 128; }
constexpr int kMmaWarp = 8;    // MMA issuer of softmax warpgroup 0, TMEM owner
constexpr int kLoadWarp = 9;   // TMA producer
constexpr int kMmaWarp1 = 10;  // MMA issuer of softmax warpgroup 1
constexpr int kTmemCols = 512;

// TMEM columns (fp32 S and O, packed 16-bit P). D = 128: S0 [0,128) S1 [128,256)
// O0 [256,384) O1 [384,512), and P_w overwrites the first half of S_w. D = 64: P has
// columns of its own, S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384) O0 [384,448)
// O1 [448,512), which lets the next S of a warpgroup be computed while its softmax still
// runs (see the MMA schedule).
template <int D>
struct TmemCols {
  static constexpr bool kSepP = (D == 64);
  __host__ __device__ static constexpr uint32_t s(int w) { return static_cast<uint32_t>(w * kBN); }
  __host__ __device__ static constexpr uint32_t p(int w) { return static_cast<uint32_t>(kSepP ? 2 * kBN + w * (kBN / 2) : w * kBN); }
  __host__ __device__ static constexpr uint32_t o(int w) { return static_cast<uint32_t>(kSepP ? 3 * kBN + w * D : 2 * kBN + w * D); }
};
static_assert(TmemCols<64>::o(1) + 64 <= kTmemCols && TmemCols<128>::o(1) + 128 <= kTmemCols, "TMEM budget");
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;

__host__ __device__ constexpr int item_rows(bool splitk) { return splitk ? kBM : 2 * kBM; }

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
  int num_mb;                  // row blocks per head: ceil(N / item_rows)
  int num_items;               // BH * num_mb
  int section;                 // causal ordering: heads per L2 section
  // Work items per CTA, or nullptr for the persistent snake order: gridDim.x + 1 offsets, then
  // the item indices of CTA c at [offsets[c], offsets[c + 1]) (device memory, read only).
  const int* schedule;
  float scale_log2;            // scale * log2(e)
  int force_stall;             // test hook: the MMA warp first waits on a barrier nothing arrives on
  // Split-KV partial form only: the K/V tiles of every query tile are divided into num_splits
  // contiguous ranges, one work item each; item results go to o_part [num_splits, BH, N, D]
  // and lse_part [num_splits, BH, N] (fp32) instead of O and lse.
  int num_splits;
  float* o_part;
  float* lse_part;
  CUtensorMap tm_op;  // o_part as 3-D fp32 (D, N, num_splits * BH), box (32, 32, 1), 128B swizzle
};

// kRingInQ1: single-query-tile items leave the second Q tile unused, and the K/V ring starts
// there, one stage deeper. kHalfStaging (two-query-tile
// items): at D = 128 each warpgroup stages one 64-column chunk of O at a time, and the space
// saved is a fourth K/V stage.
template <int D, bool kRingInQ1 = false, bool kHalfStaging = false>
struct SmemLayout {
  static constexpr int kChunks = D / 64;           // 64-column (128-byte) swizzle chunks per row
  static constexpr int kChunkBytes = kBM * 128;    // one chunk of a 128-row tile
  static constexpr int kTileBytes = kBM * D * 2;   // a 128 x D fp16/bf16 tile
  static constexpr bool kOneChunkStaging = kHalfStaging && kChunks > 1;
  static constexpr int kStages = ((D == 64) ? 8 : 3) + (kRingInQ1 ? 1 : 0) + (kOneChunkStaging ? 1 : 0);
  static constexpr int kOStageBytes = kOneChunkStaging ? kChunkBytes : kTileBytes;  // per warpgroup
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + (kRingInQ1 ? 1 : 2) * kTileBytes;
  static constexpr int kOOff = kKVOff + kStages * kTileBytes;  // two staging areas for O
  static constexpr int kBarOff = kOOff + 2 * kOStageBytes;
  // barrier indices
  static constexpr int kQFull = 0;
  static constexpr int kQEmpty = 1;
  static constexpr int kKVFull = 2;
  static constexpr int kKVEmpty = kKVFull + kStages;
  static constexpr int kSFull = kKVEmpty + kStages;  // [2] S of warpgroup i is in TMEM
  static constexpr int kPFull = kSFull + 2;          // [2] P of warpgroup i is in TMEM
  static constexpr int kOFull = kPFull + 2;          // [2] last PV of warpgroup i completed
  static constexpr int kSFree = kOFull + 2;          // [2] warpgroup i has read its S (separate-P form)
  static constexpr int kPVDone = kSFree + 2;         // [2] each PV of warpgroup i completed (separate-P form)
  static constexpr int kStats = kPVDone + 2;         // split-K: warpgroup 1 published (m, l)
  static constexpr int kO1Free = kStats + 1;         // split-K: warpgroup 0 finished reading O1
  static constexpr int kO1Self = kO1Free + 1;        // paired: warpgroup 1 finished reading O1 for its own store
  static constexpr int kOFullB = kO1Self + 1;        // paired: last PV of warpgroup 1's own query tile completed
  static constexpr int kStall = kOFullB + 1;         // never arrived on (watchdog test hook)
  static constexpr int kDrain = kStall + 1;          // [2] per MMA warp
  static constexpr int kNumBars = kDrain + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kStatsOff = kMiscOff + 16;  // split-K (m, l) hand-off, 2 x 128 fp32
  static constexpr int kBytes = kStatsOff + 2 * kBM * 4;
  static constexpr int kDynamicBytes = kBytes + 1024;  // slack to align the base to 1024 bytes
  static_assert(kDynamicBytes <= 232448, "shared memory budget");
};

// Layout of a kernel instance. Single-query-tile items run the ring into the unused second
// Q tile; two-query-tile items and paired split-K units hold two Q tiles and, at D = 128,
// stage O one chunk at a time.
template <int D, bool SPLITK, bool PAIR>
using KernelLayout = SmemLayout<D, SPLITK && !PAIR, !SPLITK || PAIR>;

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
  int mb;     // row block: 256 rows (two query tiles) or, split-K, one 128-row query tile
  int split;  // split-KV partial form: which K/V range of the query tile
};

// Work-item order. Non-causal: head-major (all row blocks of a head run close together, so
// the head's K/V is read from DRAM about once). Causal: heads are grouped into sections that
// fit in L2; inside a section the most expensive row blocks (largest mb) come first.
template <bool CAUSAL>
__host__ __device__ inline Item decode_item(int t, const Params& p) {
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

// Per work item: nk = K/V tiles loaded, n[w] = K/V tiles processed by warpgroup w (0 = idle).
template <bool CAUSAL, bool SPLITK>
__host__ __device__ inline void tile_counts(int mb, int N, int& nk, int& n0, int& n1) {
  const int nkt = (N + kBN - 1) / kBN;
  if (SPLITK) {
    nk = CAUSAL ? min(mb + 1, nkt) : nkt;
    n0 = (nk + 1) >> 1;
    n1 = nk >> 1;
  } else {
    const bool t1 = mb * 2 * kBM + kBM < N;
    if (CAUSAL) {
      n0 = min(2 * mb + 1, nkt);
      n1 = t1 ? min(2 * mb + 2, nkt) : 0;
    } else {
      n0 = nkt;
      n1 = t1 ? nkt : 0;
    }
    nk = max(n0, n1);
  }
}

// Work item t: its query rows and its K/V tiles [jb, jb + nk), of which warpgroup w processes
// n_w (tile_counts). In the split-KV partial form item t is split t % num_splits of row block
// t / num_splits, whose nk_full tiles are divided as [s nk_full / S, (s + 1) nk_full / S): a
// range may be empty (nk = 0) when the row block has fewer tiles than splits.
template <bool CAUSAL, bool SPLITK, bool PARTIAL>
__device__ __forceinline__ Item decode_work(int t, const Params& p, int& jb, int& nk, int& n0, int& n1) {
  int s = 0;
  if (PARTIAL) {
    s = t % p.num_splits;
    t /= p.num_splits;
  }
  Item it = decode_item<CAUSAL>(t, p);
  it.split = s;
  tile_counts<CAUSAL, SPLITK>(it.mb, p.N, nk, n0, n1);
  jb = 0;
  if (PARTIAL) {
    const int lo = s * nk / p.num_splits;
    const int hi = (s + 1) * nk / p.num_splits;
    jb = lo;
    nk = hi - lo;
    n0 = (nk + 1) >> 1;
    n1 = nk >> 1;
  }
  return it;
}

// k-th work item of this CTA (-1 when done): from the schedule when there is one, else in
// snake order over the sorted item list (with one CTA per item, just blockIdx.x).
__device__ __forceinline__ int item_of(int k, const Params& p) {
  if (p.schedule != nullptr) {
    const int b = __ldg(p.schedule + blockIdx.x) + k;
    return b < __ldg(p.schedule + blockIdx.x + 1) ? __ldg(p.schedule + gridDim.x + 1 + b) : -1;
  }
  const int num_items = p.num_items;
  const int G = gridDim.x;
  const long long base = static_cast<long long>(k) * G;
  if (base >= num_items) return -1;
  const int c = (k & 1) ? (G - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const long long t = base + c;
  return t < num_items ? static_cast<int>(t) : -1;
}

// The work of one pass through a CTA's loops. Two-query-tile and unpaired single-query-tile
// forms: one work item `a` (decode_work), whose K/V positions [0, nk) are its tiles jb + j;
// in the split-K form position j belongs to warpgroup j & 1 as its tile u = j >> 1.
// Paired split-K form (a launch with between one and two items per CTA): CTA c runs items c
// and 2 G - 1 - c of the sorted list together, `a` the one with more key tiles (na >= nb).
// Warpgroup 0 takes a's first n0 = ceil((na + nb) / 2) tiles; warpgroup 1 takes all nb
// tiles of b, stores b itself, then takes a's remaining n1 - nb tiles, which warpgroup 0
// merges as in the split-K form. Each warpgroup then runs n0 or n0 - 1 tiles, where two
// items one after another would run ceil(na / 2) + ceil(nb / 2) tiles and an item change.
struct Unit {
  Item a, b;
  int jb;          // first K/V tile of a's range (split-KV partial form)
  int nk;          // K/V positions: na, or na + nb when paired
  int n0, n1;      // tiles of warpgroup 0 and 1
  int nb;          // tiles of b (0: not paired)
};

// The paired unit of CTA c of G (items c and 2 G - 1 - c; false when c has no item).
template <bool CAUSAL>
__host__ __device__ inline bool pair_unit(int c, int G, const Params& p, Unit& U, int* ta_out = nullptr,
                                          int* tb_out = nullptr) {
  int ta = c, tb = 2 * G - 1 - c;
  if (ta >= p.num_items) return false;
  U.a = decode_item<CAUSAL>(ta, p);
  U.a.split = 0;
  int na, nb = 0, x0, x1;
  tile_counts<CAUSAL, true>(U.a.mb, p.N, na, x0, x1);
  if (tb < p.num_items) {
    U.b = decode_item<CAUSAL>(tb, p);
    U.b.split = 0;
    tile_counts<CAUSAL, true>(U.b.mb, p.N, nb, x0, x1);
    if (nb > na) {
      const Item t = U.a;
      U.a = U.b;
      U.b = t;
      const int n = na;
      na = nb;
      nb = n;
      const int tt = ta;
      ta = tb;
      tb = tt;
    }
  } else {
    tb = -1;
  }
  U.jb = 0;
  U.nk = na + nb;
  U.n0 = (U.nk + 1) >> 1;
  U.n1 = U.nk >> 1;
  U.nb = nb;
  if (ta_out != nullptr) *ta_out = ta;
  if (tb_out != nullptr) *tb_out = tb;
  return true;
}

template <bool CAUSAL, bool SPLITK, bool PARTIAL, bool PAIR>
__device__ __forceinline__ bool decode_unit(int k, const Params& p, Unit& U) {
  if constexpr (PAIR) {
    return k == 0 && pair_unit<CAUSAL>(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), p, U);
  } else {
    const int t = item_of(k, p);
    if (t < 0) return false;
    U.a = decode_work<CAUSAL, SPLITK, PARTIAL>(t, p, U.jb, U.nk, U.n0, U.n1);
    U.nb = 0;
    return true;
  }
}

// Split-K form: the K/V tile of warpgroup w's u-th position, and whether it is one of b's.
template <bool PAIR>
__device__ __forceinline__ int unit_tile(const Unit& U, int w, int u, bool& from_b) {
  from_b = false;
  if (!PAIR || U.nb == 0) return U.jb + 2 * u + w;
  if (w == 0) return u;
  from_b = u < U.nb;
  return from_b ? u : U.n0 + (u - U.nb);
}

template <int D, bool BF16, bool CAUSAL, bool SPLITK, bool PARTIAL, bool PAIR = false>
__global__ void __launch_bounds__(kNumThreads, 1) fa_fwd_kernel(const __grid_constant__ Params p) {
  static_assert(!PARTIAL || SPLITK, "the split-KV partial form uses one query tile per item");
  static_assert(!PAIR || (SPLITK && !PARTIAL), "pairs are formed from whole single-query-tile items");
  static_assert(!PAIR || TmemCols<D>::kSepP, "pairs use the separate-P split-K issue order (D = 64)");
  constexpr bool kRegSplit = reg_split<D>();
  // Two MMA issuers (one per softmax warpgroup) where that measured faster: D = 64 with two
  // query tiles per item (c3 43.2 -> 40.5 us). At D = 128 and with single query tiles one
  // issuer is faster (two made c4 8%, c5 10% and the short causal c2 7% slower).
  constexpr bool kDualMma = (D == 64) && !SPLITK;
  constexpr uint32_t kMmaIssuers = kDualMma ? 2 : 1;
  using L = KernelLayout<D, SPLITK, PAIR>;
  using TC = TmemCols<D>;
  constexpr bool kSepP = TC::kSepP;
  constexpr int kItemRows = item_rows(SPLITK);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](int idx) -> uint32_t { return sbase + L::kBarOff + 8u * idx; };
  auto q_addr = [&](int i) -> uint32_t { return sbase + L::kQOff + i * L::kTileBytes; };
  auto kv_addr = [&](int s) -> uint32_t { return sbase + L::kKVOff + s * L::kTileBytes; };
  auto o_addr = [&](int i) -> uint32_t { return sbase + L::kOOff + i * L::kOStageBytes; };
  float* stats_m = reinterpret_cast<float*>(smem + L::kStatsOff);
  float* stats_l = stats_m + kBM;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const Watch watch{abort_flag, p.status, p.timeout_ns};

  // Q tiles of unit Uq into the Q buffers (two query tiles of one item, or, paired, a's then b's).
  auto load_q = [&](const Unit& Uq) {
    const int nq = (SPLITK ? Uq.nb > 0 : Uq.n1 > 0) ? 2 : 1;
    mbar_arrive_expect_tx(bar(L::kQFull), nq * L::kTileBytes);
    for (int i = 0; i < nq; ++i) {
      const Item& qi = (SPLITK && i > 0) ? Uq.b : Uq.a;
      const int row0 = SPLITK ? qi.mb * kBM : qi.mb * kItemRows + i * kBM;
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_3d(q_addr(i) + c * L::kChunkBytes, &p.tm_q, bar(L::kQFull), c * 64, row0, qi.bh);
    }
  };
  // Setup. The producer lane initialises the barriers, decodes its first work unit (kernel
  // parameters and the work table, copied before the launch in stream order) and, once the
  // previous kernel on the stream is done, loads that unit's Q tiles, all before the CTA-wide
  // barrier: the first load leaves while the other warps set up.
  Unit u_first{};
  bool u_first_ok = false, q_first = false;
  if (warp == kLoadWarp && lane == 0) {
    mbar_init(bar(L::kQFull), 1);
    mbar_init(bar(L::kQEmpty), kMmaIssuers);  // one arrival per MMA warp
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kKVFull + s), 1);
      mbar_init(bar(L::kKVEmpty + s), kMmaIssuers);  // one release per MMA warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kSFull + i), 1);
      mbar_init(bar(L::kPFull + i), kBM);
      mbar_init(bar(L::kOFull + i), 1);
      mbar_init(bar(L::kSFree + i), kBM);
      mbar_init(bar(L::kPVDone + i), 1);
    }
    mbar_init(bar(L::kStats), kBM);
    mbar_init(bar(L::kO1Free), kBM);
    mbar_init(bar(L::kO1Self), kBM);
    mbar_init(bar(L::kOFullB), 1);
    mbar_init(bar(L::kStall), 1);
    mbar_init(bar(L::kDrain), 1);
    mbar_init(bar(L::kDrain + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&p.tm_q);
    prefetch_tmap(&p.tm_k);
    prefetch_tmap(&p.tm_v);
    prefetch_tmap(&p.tm_o);
    u_first_ok = decode_unit<CAUSAL, SPLITK, PARTIAL, PAIR>(0, p, u_first);
    if (u_first_ok && u_first.nk > 0) {
      grid_dependency_wait();  // the inputs may be written by the previous kernel on the stream
      load_q(u_first);         // fresh Q buffers: no wait for an earlier reader
      q_first = true;
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // Everything above touched only this CTA's shared memory and TMEM; the inputs may be
  // written by the previous kernel on the stream.
  grid_dependency_wait();

  if (warp >= 8) {
    if constexpr (kRegSplit) regs_lower<kOtherRegs>();
    if (warp == kLoadWarp) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        uint32_t kv_pos = 0, q_loads = 0;
        bool ok = true;
        Unit U{};
        // K/V tile of position j of the current unit into the next ring slot.
        auto load_kv = [&](const void* tm, int j) -> bool {
          int jt = U.jb + j, bh = U.a.bh;
          if (SPLITK) {
            bool from_b;
            jt = unit_tile<PAIR>(U, j & 1, j >> 1, from_b);
            if (from_b) bh = U.b.bh;
          }
          const uint32_t s = kv_pos % L::kStages;
          if (!wait_phase(bar(L::kKVEmpty + s), ((kv_pos / L::kStages) & 1) ^ 1, watch, 1)) return false;
          mbar_arrive_expect_tx(bar(L::kKVFull + s), L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(kv_addr(s) + c * L::kChunkBytes, tm, bar(L::kKVFull + s), c * 64, jt * kBN, bh);
          ++kv_pos;
          return true;
        };
        for (int k = 0; ok; ++k) {
          if (k == 0) {
            if (!u_first_ok) break;
            U = u_first;
          } else if (!decode_unit<CAUSAL, SPLITK, PARTIAL, PAIR>(k, p, U)) {
            break;
          }
          const int nk = U.nk;
          if (nk == 0) continue;  // empty split-KV range: nothing to load
          if (!(k == 0 && q_first)) {  // the first unit's Q tiles left during setup
            // Q tiles: wait until every S MMA of the previous item has read them.
            if (!(ok = wait_phase(bar(L::kQEmpty), (q_loads & 1) ^ 1, watch, 0))) break;
            load_q(U);
          }
          ++q_loads;
          // K/V in the MMA warp's consumption order:
          //   two query tiles, P in S's columns:   K0 V0 K1 V1 K2 ...
          //   two query tiles, separate P, and
          //   split-K, P in S's columns:           K0 K1 V0 K2 V1 K3 V2 ...
          //   split-K, separate P:                 K0 K1 K2 K3 V0 V1 K4 K5 V2 V3 ...
          if (!SPLITK && !kSepP) {
            for (int j = 0; j < nk && ok; ++j) ok = load_kv(&p.tm_k, j) && load_kv(&p.tm_v, j);
          } else if (SPLITK && kSepP) {
            ok = load_kv(&p.tm_k, 0);
            if (nk > 1) ok = ok && load_kv(&p.tm_k, 1);
            for (int t2 = 0; t2 < nk && ok; t2 += 2) {
              if (t2 + 2 < nk) ok = ok && load_kv(&p.tm_k, t2 + 2);
              if (t2 + 3 < nk) ok = ok && load_kv(&p.tm_k, t2 + 3);
              ok = ok && load_kv(&p.tm_v, t2);
              if (t2 + 1 < nk) ok = ok && load_kv(&p.tm_v, t2 + 1);
            }
          } else {
            ok = load_kv(&p.tm_k, 0);
            for (int j = 0; j < nk && ok; ++j) {
              if (j + 1 < nk) ok = load_kv(&p.tm_k, j + 1);
              ok = ok && load_kv(&p.tm_v, j);
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
    } else if (kDualMma && (warp == kMmaWarp || warp == kMmaWarp1)) {
      // ------------------------------------------------------------ MMA issuers (dual, D = 64, two query tiles)
      // Warp kMmaWarp issues every MMA of softmax warpgroup 0 (its S and its PV), warp
      // kMmaWarp1 those of warpgroup 1. Issuing a tcgen05.mma blocks the warp for about the
      // MMA's tensor time, so one issuer would leave the tensor pipe idle whenever it waited
      // for one warpgroup; with one issuer per warpgroup, the other one keeps the pipe fed.
      // Both walk every K/V ring position in the producer's order (waiting for each one, so no
      // phase can be mistaken for a later one) and release every position: with a commit where
      // they used it, with a plain arrive where the tile belongs to the other warpgroup. A stage
      // is free once both released it. The whole warp runs the loop; one elected lane issues.
      {
        const int w = warp == kMmaWarp ? 0 : 1;  // the warpgroup this warp serves
        const uint32_t leader = elect_one_lane();
        constexpr uint32_t idesc_s = instr_desc_f16(BF16, kBM, kBN, false);
        constexpr uint32_t idesc_o = instr_desc_f16(BF16, kBM, D, true);
        uint32_t kv_pos = 0, items = 0, merges = 0, pcnt = 0, tiles_w = 0;
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t parity, unsigned site) {
          return __all_sync(0xffffffffu, wait_phase(b, parity, watch, site));
        };
        // Next K/V ring slot: wait until TMA has filled it; returns its stage.
        auto next_slot = [&](uint32_t& stage) -> bool {
          stage = kv_pos % L::kStages;
          if (!wait(bar(L::kKVFull + stage), (kv_pos / L::kStages) & 1, 3)) return false;
          ++kv_pos;
          tc_fence_after();
          return true;
        };
        auto release = [&](uint32_t stage) { mma_commit_leader(bar(L::kKVEmpty + stage), leader); };
        auto pass = [&](uint32_t stage) {  // a position this warpgroup does not use
          if (leader) mbar_arrive(bar(L::kKVEmpty + stage));
        };

        // Descriptors are built once; per stage / tile / k-step only the 14-bit start-address
        // field (address >> 4, no carry possible below 256 KB) is advanced.
        const uint64_t q_desc = smem_desc_sw128(q_addr(0), 16, 1024);
        const uint64_t k_desc = smem_desc_sw128(kv_addr(0), 16, 1024);
        const uint64_t v_desc = smem_desc_sw128(kv_addr(0), L::kChunkBytes, 1024);
        constexpr uint32_t kTileEnc = L::kTileBytes >> 4;

        // S_w = Q_qi K^T into TMEM columns [128 w, 128 w + 128). Q is released (one of the two
        // arrivals kQEmpty needs) once this warpgroup's last S MMA of the item has been issued.
        int s_left = 0;  // S MMAs of the current item not yet issued for this warpgroup
        auto issue_s = [&](int qi, uint32_t stage) {
          const uint32_t d_tmem = tmem + TC::s(w);
          const uint64_t a0 = q_desc + static_cast<uint32_t>(qi) * kTileEnc;
          const uint64_t b0 = k_desc + stage * kTileEnc;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss_leader(d_tmem, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u, leader);
          }
          mma_commit_leader(bar(L::kSFull + w), leader);
          if (--s_left == 0) mma_commit_leader(bar(L::kQEmpty), leader);
        };
        // O_w (+)= P_w V; P_w is 64 columns of packed fp16/bf16 pairs (TmemCols).
        // V tile: keys are the K dimension (rows, 128 B apart), D is the N dimension (MN-major):
        // 8-key groups are 1024 B apart, 64-column chunks kChunkBytes apart (the LBO).
        auto issue_pv = [&](uint32_t stage, bool accumulate, bool last) -> bool {
          if (!wait(bar(L::kPFull + w), pcnt & 1, 5 + w)) return false;
          ++pcnt;
          tc_fence_after();
          const uint32_t d_tmem = tmem + TC::o(w);
          const uint32_t a_tmem = tmem + TC::p(w);
          const uint64_t b0 = v_desc + stage * kTileEnc;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_leader(d_tmem, a_tmem + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc_o,
                          (accumulate || kk > 0) ? 1u : 0u, leader);
          if (kSepP) mma_commit_leader(bar(L::kPVDone + w), leader);
          if (last) mma_commit_leader(bar(L::kOFull + w), leader);
          return true;
        };
        // Separate-P form: the warpgroup signals kSFree once per tile it processes, so the
        // hand-back of its tile u of the current item is completion tiles_w + u + 1.
        auto wait_s_free = [&](int u) -> bool {
          const uint32_t c = tiles_w + static_cast<uint32_t>(u) + 1;
          if (!wait(bar(L::kSFree + w), (c - 1) & 1, 14 + w)) return false;
          tc_fence_after();
          return true;
        };

        if (p.force_stall) ok = wait(bar(L::kStall), 0, 12);  // runs out: exercises the abort path
        for (int k = 0; ok; ++k) {
          const int t = item_of(k, p);
          if (t < 0) break;
          int jb, nk, n0, n1;
          decode_work<CAUSAL, SPLITK, PARTIAL>(t, p, jb, nk, n0, n1);
          if (nk == 0) continue;  // empty split-KV range
          const int n_w = w ? n1 : n0;
          if (!(ok = wait(bar(L::kQFull), items & 1, 2))) break;
          s_left = n_w;
          if (n_w == 0 && leader) mbar_arrive(bar(L::kQEmpty));  // nothing of this item to issue
          // Key tile j is this warpgroup's u-th tile (or not its own).
          auto own = [&](int j, int& u) -> bool {
            if (SPLITK) {
              u = j >> 1;
              return (j & 1) == w;
            }
            u = j;
            return j < n_w;
          };
          auto on_k = [&](int j) -> bool {
            uint32_t st;
            if (!next_slot(st)) return false;
            int u;
            if (!own(j, u)) {
              pass(st);
              return true;
            }
            // With separate P the next S only needs the previous S read; otherwise it follows the
            // PV that read P (same columns) in this warp's in-order issue.
            if (kSepP && u > 0 && !wait_s_free(u - 1)) return false;
            issue_s(SPLITK ? 0 : w, st);
            release(st);
            return true;
          };
          auto on_v = [&](int j) -> bool {
            uint32_t st;
            if (!next_slot(st)) return false;
            int u;
            if (!own(j, u)) {
              pass(st);
              return true;
            }
            // Warpgroup 1's O is overwritten by its first PV: the previous merge must have read it.
            if (SPLITK && w == 1 && u == 0 && merges > 0 && !wait(bar(L::kO1Free), (merges - 1) & 1, 13))
              return false;
            if (!issue_pv(st, u > 0, u == n_w - 1)) return false;
            release(st);
            return true;
          };
          // The producer's order (see the producer).
          if (!SPLITK && !kSepP) {
            for (int j = 0; j < nk && ok; ++j) ok = on_k(j) && on_v(j);
          } else if (SPLITK && kSepP) {
            ok = on_k(0);
            if (ok && nk > 1) ok = on_k(1);
            for (int t2 = 0; t2 < nk && ok; t2 += 2) {
              if (t2 + 2 < nk) ok = on_k(t2 + 2);
              if (ok && t2 + 3 < nk) ok = on_k(t2 + 3);
              ok = ok && on_v(t2);
              if (ok && t2 + 1 < nk) ok = on_v(t2 + 1);
            }
          } else {
            ok = on_k(0);
            for (int j = 0; j < nk && ok; ++j) {
              if (j + 1 < nk) ok = on_k(j + 1);
              ok = ok && on_v(j);
            }
          }
          if (!ok) break;
          if (SPLITK && w == 1 && n1 > 0) ++merges;
          ++items;
          tiles_w += static_cast<uint32_t>(n_w);
        }
        // Whatever happened, wait for every MMA this warp issued before TMEM can be freed.
        mma_commit_leader(bar(L::kDrain + w), leader);
        if (leader) wait_phase_drain(bar(L::kDrain + w), 0);
      }
      __syncwarp();
    } else if (!kDualMma && warp == kMmaWarp) {
      // ------------------------------------------------------------ MMA issuer (single)
      // One warp issues the MMAs of both softmax warpgroups (D = 128 and single-query-tile items).
      // The whole warp runs this loop; one elected lane issues each tcgen05 instruction.
      {
        const uint32_t leader = elect_one_lane();
        constexpr uint32_t idesc_s = instr_desc_f16(BF16, kBM, kBN, false);
        constexpr uint32_t idesc_o = instr_desc_f16(BF16, kBM, D, true);
        uint32_t kv_pos = 0, items = 0;
        uint32_t pcnt0 = 0, pcnt1 = 0;  // P hand-offs consumed per warpgroup
        bool ok = true;
        auto wait = [&](uint32_t b, uint32_t parity, unsigned site) {
          return __all_sync(0xffffffffu, wait_phase(b, parity, watch, site));
        };
        // Next K/V ring slot: wait until TMA has filled it; returns its stage.
        auto next_slot = [&](uint32_t& stage) -> bool {
          stage = kv_pos % L::kStages;
          if (!wait(bar(L::kKVFull + stage), (kv_pos / L::kStages) & 1, 3)) return false;
          ++kv_pos;
          tc_fence_after();
          return true;
        };

        // Descriptors are built once; per stage / tile / k-step only the 14-bit start-address
        // field (address >> 4, no carry possible below 256 KB) is advanced.
        const uint64_t q_desc = smem_desc_sw128(q_addr(0), 16, 1024);
        const uint64_t k_desc = smem_desc_sw128(kv_addr(0), 16, 1024);
        const uint64_t v_desc = smem_desc_sw128(kv_addr(0), L::kChunkBytes, 1024);
        constexpr uint32_t kTileEnc = L::kTileBytes >> 4;

        // S_w = Q_qi K^T into TMEM columns [128 w, 128 w + 128).
        // Q is released as soon as the item's last S MMA has been issued (its completion then
        // covers every MMA that reads Q), so the next item's Q load overlaps this item's tail.
        int s_left = 0;  // S MMAs of the current item not yet issued
        auto issue_s = [&](int w, int qi, uint32_t stage) {
          const uint32_t d_tmem = tmem + TC::s(w);
          const uint64_t a0 = q_desc + static_cast<uint32_t>(qi) * kTileEnc;
          const uint64_t b0 = k_desc + stage * kTileEnc;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ss_leader(d_tmem, a0 + off, b0 + off, idesc_s, kk > 0 ? 1u : 0u, leader);
          }
          mma_commit_leader(bar(L::kSFull + w), leader);
          if (--s_left == 0) mma_commit_leader(bar(L::kQEmpty), leader);
        };
        // O_w (+)= P_w V; P_w is 64 columns of packed fp16/bf16 pairs (TmemCols).
        // V tile: keys are the K dimension (rows, 128 B apart), D is the N dimension (MN-major):
        // 8-key groups are 1024 B apart, 64-column chunks kChunkBytes apart (the LBO).
        auto issue_pv = [&](int w, uint32_t stage, bool accumulate, bool last) -> bool {
          const uint32_t pc = w ? pcnt1 : pcnt0;
          if (!wait(bar(L::kPFull + w), pc & 1, 5 + w)) return false;
          if (w) ++pcnt1;
          else ++pcnt0;
          tc_fence_after();
          const uint32_t d_tmem = tmem + TC::o(w);
          const uint32_t a_tmem = tmem + TC::p(w);
          const uint64_t b0 = v_desc + stage * kTileEnc;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_leader(d_tmem, a_tmem + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc_o,
                          (accumulate || kk > 0) ? 1u : 0u, leader);
          if (kSepP) mma_commit_leader(bar(L::kPVDone + w), leader);
          if (last) mma_commit_leader(bar(L::kOFull + w), leader);
          return true;
        };
        // The same with the barrier to commit after the PV chosen by the caller (0: none), for
        // the split-K form at D = 64, where a pair's b ends on a barrier of its own. The other
        // paths keep the constant-barrier form: passing the barrier for every PV made the long
        // D = 128 split-K chains 4-5% slower (c5, lc1).
        auto issue_pv_to = [&](int w, uint32_t stage, bool accumulate, uint32_t done_bar) -> bool {
          const uint32_t pc = w ? pcnt1 : pcnt0;
          if (!wait(bar(L::kPFull + w), pc & 1, 5 + w)) return false;
          if (w) ++pcnt1;
          else ++pcnt0;
          tc_fence_after();
          const uint32_t d_tmem = tmem + TC::o(w);
          const uint32_t a_tmem = tmem + TC::p(w);
          const uint64_t b0 = v_desc + stage * kTileEnc;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_leader(d_tmem, a_tmem + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc_o,
                          (accumulate || kk > 0) ? 1u : 0u, leader);
          if (kSepP) mma_commit_leader(bar(L::kPVDone + w), leader);
          if (done_bar != 0) mma_commit_leader(done_bar, leader);
          return true;
        };
        // Split-K: warpgroup 1's O1 is overwritten by the first PV of each of its accumulations
        // (an item's odd tiles; paired, b's tiles, then a's remaining ones), so whoever read the
        // previous one must be done: warpgroup 0's merge (kO1Free) or, paired, warpgroup 1's
        // own store (kO1Self). Both barriers complete once per such read, in order.
        uint32_t merges = 0, selfs = 0;  // accumulations into O1 issued, by their reader
        int o1_reader = 0;               // reader of the last one: 0 none, 1 merge, 2 own store
        auto o1_begin = [&](bool own_b) -> bool {
          if (o1_reader == 1 && !wait(bar(L::kO1Free), (merges - 1) & 1, 13)) return false;
          if (o1_reader == 2 && !wait(bar(L::kO1Self), (selfs - 1) & 1, 13)) return false;
          if (own_b) {
            ++selfs;
            o1_reader = 2;
          } else {
            ++merges;
            o1_reader = 1;
          }
          return true;
        };
        // Separate-P form: warpgroup w signals kSFree once per tile it processes (also for its
        // last tile of an item, which has no next S), so the waits name the completion they need:
        // the hand-back of tile u of the current item is completion tiles_w + u + 1, where tiles_w
        // counts warpgroup w's tiles in earlier items.
        uint32_t tiles0 = 0, tiles1 = 0;
        auto wait_s_free = [&](int w, int u) -> bool {
          const uint32_t c = (w ? tiles1 : tiles0) + static_cast<uint32_t>(u) + 1;
          if (!wait(bar(L::kSFree + w), (c - 1) & 1, 14 + w)) return false;
          tc_fence_after();
          return true;
        };
        auto release = [&](uint32_t stage) { mma_commit_leader(bar(L::kKVEmpty + stage), leader); };

        if (p.force_stall) ok = wait(bar(L::kStall), 0, 12);  // runs out: exercises the abort path
        for (int k = 0; ok; ++k) {
          Unit U;
          if (!decode_unit<CAUSAL, SPLITK, PARTIAL, PAIR>(k, p, U)) break;
          const int nk = U.nk, n0 = U.n0, n1 = U.n1;
          if (nk == 0) continue;  // empty split-KV range
          s_left = SPLITK ? nk : n0 + n1;
          if (!(ok = wait(bar(L::kQFull), items & 1, 2))) break;
          uint32_t sk, sv;
          // Split-K: Q tile read by warpgroup w's u-th S (paired: b's tile is the second one).
          auto q_of = [&](int w, int u) -> int { return (PAIR && w == 1 && u < U.nb) ? 1 : 0; };
          // Split-K PV of warpgroup w's u-th tile: opens an accumulation (and, for warpgroup 1,
          // waits until O1 is free) or adds to it, and signals the end of one.
          auto split_pv = [&](int w, int u, uint32_t stage) -> bool {
            const bool b_end = PAIR && w == 1 && u == U.nb - 1;
            const bool start = u == 0 || (PAIR && w == 1 && U.nb > 0 && u == U.nb);
            if (w == 1 && start && !o1_begin(PAIR && u < U.nb)) return false;
            const uint32_t done = b_end ? bar(L::kOFullB) : (u == (w ? n1 : n0) - 1 ? bar(L::kOFull + w) : 0u);
            return issue_pv_to(w, stage, !start, done);
          };
          if (kSepP && !SPLITK) {
            // Separate P: S_w(j+1) is issued as soon as warpgroup w has read S_w(j), before
            // PV_w(j), so the tensor core computes the next S while the softmax runs.
            if (!(ok = next_slot(sk))) break;
            issue_s(0, 0, sk);
            if (n1 > 0) issue_s(1, 1, sk);
            release(sk);
            for (int j = 0; j < nk && ok; ++j) {
              bool k_next = false;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                if (j + 1 < (w ? n1 : n0)) {
                  if (!(ok = wait_s_free(w, j))) break;
                  if (!k_next && !(ok = next_slot(sk))) break;
                  k_next = true;
                  issue_s(w, w, sk);
                }
              }
              if (!ok) break;
              if (k_next) release(sk);
              if (!(ok = next_slot(sv))) break;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int nw = w ? n1 : n0;
                if (j < nw && !(ok = issue_pv(w, sv, j > 0, j == nw - 1))) break;
              }
              if (!ok) break;
              release(sv);
            }
          } else if (kSepP && SPLITK) {
            // Separate P, one query tile: tile j belongs to warpgroup j & 1. Per round t2
            // (even tile t2, odd tile t2 + 1): next S of each warpgroup, then both PVs.
            if (!(ok = next_slot(sk))) break;
            issue_s(0, 0, sk);
            release(sk);
            if (nk > 1) {
              if (!(ok = next_slot(sk))) break;
              issue_s(1, q_of(1, 0), sk);
              release(sk);
            }
            for (int t2 = 0; t2 < nk && ok; t2 += 2) {
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                if (t2 + 2 + w < nk) {
                  if (!(ok = wait_s_free(w, t2 >> 1)) || !(ok = next_slot(sk))) break;
                  issue_s(w, q_of(w, (t2 >> 1) + 1), sk);
                  release(sk);
                }
              }
              if (!ok) break;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                if (t2 + w < nk) {
                  if (!(ok = next_slot(sv))) break;
                  if (!(ok = split_pv(w, t2 >> 1, sv))) break;
                  release(sv);
                }
              }
            }
          } else if (!SPLITK) {
            // Both query tiles against K0, then per K/V tile j: PV_w(j) and S_w(j+1), w = 0, 1.
            if (!(ok = next_slot(sk))) break;
            issue_s(0, 0, sk);
            if (n1 > 0) issue_s(1, 1, sk);
            release(sk);
            for (int j = 0; j < nk && ok; ++j) {
              if (!(ok = next_slot(sv))) break;
              bool k_next = false;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                const int nw = w ? n1 : n0;
                if (j < nw && !(ok = issue_pv(w, sv, j > 0, j == nw - 1))) break;
                // V_j is released right after its last PV, not after the S MMAs that follow,
                // so the producer refills the ring a step sooner (c4 206 -> 194 us).
                if (w == 1 ? j < n1 : j >= n1) release(sv);
                if (j + 1 < nw) {
                  if (!k_next && !(ok = next_slot(sk))) break;
                  k_next = true;
                  issue_s(w, w, sk);
                }
              }
              if (!ok) break;
              if (k_next) release(sk);
            }
          } else {
            // One query tile; K/V tile j belongs to warpgroup j & 1 (P in S's columns: D = 128,
            // never paired).
            //   S_0(K0), S_1(K1), then per j: PV_{j&1}(V_j), S_{j&1}(K_{j+2}).
            if (!(ok = next_slot(sk))) break;
            issue_s(0, 0, sk);
            release(sk);
            if (nk > 1) {
              if (!(ok = next_slot(sk))) break;
              issue_s(1, 0, sk);
              release(sk);
            }
            for (int j = 0; j < nk && ok; ++j) {
              const int w = j & 1;
              if (!(ok = next_slot(sv))) break;
              // O1 is overwritten by the first PV of warpgroup 1: the previous item's merge
              // must have read it.
              if (j == 1 && merges > 0 && !(ok = wait(bar(L::kO1Free), (merges - 1) & 1, 13))) break;
              if (!(ok = issue_pv(w, sv, j >= 2, j + 2 >= nk))) break;
              release(sv);
              if (j + 2 < nk) {
                if (!(ok = next_slot(sk))) break;
                issue_s(w, 0, sk);
                release(sk);
              }
            }
            if (ok && n1 > 0) ++merges;
          }
          if (!ok) break;
          ++items;
          tiles0 += static_cast<uint32_t>(n0);
          tiles1 += static_cast<uint32_t>(n1);
        }
        // Whatever happened, wait for every issued MMA before TMEM can be freed.
        mma_commit_leader(bar(L::kDrain), leader);
        if (leader) wait_phase_drain(bar(L::kDrain), 0);
      }
      __syncwarp();
    }  // the remaining warps of this warpgroup: idle
  } else {
    if constexpr (kRegSplit) regs_raise<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;        // warpgroup: query tile (two-tile items) or K parity (split-K)
    const int wq = warp & 3;         // TMEM lane quarter accessible to this warp
    const int r = wq * 32 + lane;    // row within the query tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + TC::s(wg);
    const uint32_t t_p = tmem + lane_off + TC::p(wg);
    const uint32_t t_o = tmem + lane_off + TC::o(wg);
    const uint32_t t_o1 = tmem + lane_off + TC::o(1);
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, ocnt = 0, o1cnt = 0, mcnt = 0;
    uint32_t p_sent = 0;  // P hand-offs made by this warpgroup = PVs issued for it
    bool ok = true;

    for (int k = 0; ok; ++k) {
      Unit U;
      if (!decode_unit<CAUSAL, SPLITK, PARTIAL, PAIR>(k, p, U)) break;
      const int nk = U.nk, n1 = U.n1;
      const int n_mine = wg == 0 ? U.n0 : U.n1;
      if (PARTIAL && nk == 0) {
        // Empty K/V range: the partial result has no key (lse = -inf; the merge skips it).
        const int row = U.a.mb * kBM + r;
        if (wg == 0 && row < p.N)
          p.lse_part[(static_cast<long long>(U.a.split) * p.BH + U.a.bh) * p.N + row] = -INFINITY;
        continue;
      }
      if (n_mine == 0) continue;
      // One accumulation over this warpgroup's tiles, except for warpgroup 1 of a pair: b's
      // tiles [0, nb), which it stores itself, then a's remaining tiles (if any).
      const bool two_acc = PAIR && wg == 1 && U.nb > 0;
      const int nseg = (two_acc && n1 > U.nb) ? 2 : 1;
      for (int seg = 0; seg < nseg; ++seg) {
        const bool own_b = two_acc && seg == 0;
        const int u0 = seg == 0 ? 0 : U.nb;
        const int u1 = own_b ? U.nb : n_mine;
        const Item it = own_b ? U.b : U.a;
        const int qt = SPLITK ? it.mb : 2 * it.mb + wg;  // query tile index (its diagonal K tile)
        const int row = qt * kBM + r;                     // query index within the sequence
        float m_used = -INFINITY;
        float l_run = 0.f;

        for (int jj = u0; jj < u1; ++jj) {
          int j = jj;  // K/V tile index
          if (SPLITK) {
            bool from_b;
            j = unit_tile<PAIR>(U, wg, jj, from_b);
          }
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
          if (kSepP) {
            // S is in registers: hand its TMEM columns back so the next S can be computed.
            tc_fence_before();
            mbar_arrive(bar(L::kSFree + wg));
          }
          bool abort_now = false;

          const int col0 = j * kBN;
          const bool diag = CAUSAL && j == qt;
          if (diag || col0 + kBN > p.N) {
            int lim = p.N - 1 - col0;
            if (diag) lim = min(lim, row - col0);
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c > lim) s[c] = -INFINITY;
          }
          // p = 2^(s * scale * log2 e - m) for the 64 columns of half h, packed to fp16/bf16
          // pairs and stored as P over the first half of this tile's TMEM columns (P column c
          // holds elements 2c, 2c+1; S is already in registers). Returns the half's row sum;
          // four partial sums keep the dependency chains short.
          auto exp_half = [&](float m, int h) -> float {
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m, -m);
            uint64_t acc[4] = {0, 0, 0, 0};
            uint32_t pk[kBN / 4];
#pragma unroll
            for (int i = 0; i < kBN / 4; ++i) {
              const int c = h * (kBN / 4) + i;  // column pair
              const uint64_t x2 = f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl2x2, negm2);
              float x0, x1;
              f2_unpack(x2, x0, x1);
              const float p0 = ex2_approx(x0);
              const float p1 = ex2_approx(x1);
              acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
              pk[i] = pack2<BF16>(p0, p1);
            }
            if (kSepP && h == 0 && p_sent > 0) {
              // P has columns of its own: the previous PV must have read them (and finished
              // with O) before they are overwritten.
              const bool pv_ok = wait_phase(bar(L::kPVDone + wg), (p_sent - 1) & 1, watch, 15);
              if (!__all_sync(0xffffffffu, pv_ok)) abort_now = true;
              tc_fence_after();
            }
            tmem_st32x32b_x32(t_p + h * (kBN / 4), pk);
            float a0, a1, b0, b1, c0, c1, d0, d1;
            f2_unpack(acc[0], a0, a1);
            f2_unpack(acc[1], b0, b1);
            f2_unpack(acc[2], c0, c1);
            f2_unpack(acc[3], d0, d1);
            return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
          };
          // Row max of the raw scores (scale > 0, so it commutes with the scaling), in eight
          // independent chains of 3-input max.
          auto row_max = [&]() -> float {
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
            for (int c = 16; c < kBN; c += 16)
#pragma unroll
              for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], s[c + 2 * i], s[c + 2 * i + 1]);
            return fmaxf(fmaxf(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5])), fmaxf(mx[6], mx[7]));
          };
          // Tile max first, then the exponentials against the running max m_used. m_used only
          // moves when the tile raises it by more than the threshold (then O and l are rescaled).
          const float x_max = row_max() * sl2;
          float alpha = 1.f;
          bool rescale = false;
          if (jj == u0) {
            m_used = x_max;
          } else if (x_max > m_used + kRescaleLog2) {
            alpha = ex2_approx(m_used - x_max);
            m_used = x_max;
            l_run *= alpha;
            rescale = true;
          }
          l_run += exp_half(m_used, 0) + exp_half(m_used, 1);
          if (__any_sync(0xffffffffu, rescale)) {
            // O row *= alpha (alpha = 1 for rows that keep their max). The previous PV of this
            // warpgroup has completed: with P in S's columns this tile's S was issued after it;
            // with separate P the kPVDone wait above covered it.
            if constexpr (D == 128) {
              // The whole row in one TMEM round trip (the S registers are free by now) instead of
              // four: on the long-sequence workload (scores x4) the row max keeps creeping up and
              // ~40% of warp-tiles rescale; c5 760 -> 744 us. At D = 64 it measured 1% slower.
              uint32_t o[D];
              tmem_ld32x32b_x128(t_o, o);
              const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
              for (int e = 0; e < D; e += 2) {
                float x0, x1;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), x0, x1);
                o[e] = __float_as_uint(x0);
                o[e + 1] = __float_as_uint(x1);
              }
              tmem_st32x32b_x128(t_o, o);
            } else {
#pragma unroll 1
              for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32x32b_x32(t_o + c, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32x32b_x32(t_o + c, o);
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(L::kPFull + wg));
          ++p_sent;
          if (abort_now) {
            ok = false;
            break;
          }
        }
        if (!ok) break;

        if (SPLITK && wg == 1 && !own_b) {
          // Hand (m, l) of its K/V tiles of the item to warpgroup 0, which merges and stores.
          // The previous hand-off must have been read first (warpgroup 0 signals kO1Free).
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

        // ---------------- epilogue: O / l -> staging shared memory -> TMA store; lse
        // Each warp stages and stores its own 32 rows, so no barrier spans warps.
        // (warpgroup 1 of a pair, for b: its own last-PV barrier, which only it waits on)
        bool e_ok = wait_phase(bar(own_b ? L::kOFullB : L::kOFull + wg), ocnt & 1, watch, 10 + wg);
        ++ocnt;
        const bool merge = SPLITK && wg == 0 && n1 > U.nb;
        float a_self = 1.f, a_other = 0.f;
        if (merge) {
          // Partial results of the odd tiles: O1 in TMEM, (m1, l1) from warpgroup 1.
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
          a_other = ex2_approx(m1 - m);
          l_run = l_run * a_self + l1 * a_other;
          m_used = m;
        }
        if (lane == 0) bulk_wait_group_read0();  // this warp's previous store has left the buffer
        __syncwarp();
        tc_fence_after();
        const float inv_l = 1.0f / l_run;
        const float c_self = a_self * inv_l, c_other = a_other * inv_l;
        const uint32_t ob = o_addr(wg);
        // Split-KV partial form: warp wq's fp32 boxes go to its quarter of the O staging tile of
        // warpgroup 0, then to its quarter of warpgroup 1's (which stages nothing in this form).
        auto part_box = [&](int b) -> uint32_t {
          constexpr int kPerRegion = D / 64;  // 4 KB boxes per quarter tile
          const uint32_t region = b < kPerRegion ? o_addr(0) : o_addr(1);
          return region + wq * (L::kTileBytes / 4) + (b % kPerRegion) * 4096;
        };
        // Columns per step: 64 (one 128-byte swizzle chunk) at D = 64; 32 at D = 128, where the
        // merge would otherwise hold two 64-column O rows at once.
        constexpr int kEpi = (D == 64) ? 64 : 32;
#pragma unroll 1
        for (int c = 0; c < D; c += kEpi) {
          uint32_t o[kEpi];
          if (merge) {
            uint32_t o1[kEpi];
            if constexpr (kEpi == 64) tmem_ld32x32b_x64_pair(t_o + c, t_o1 + c, o, o1);
            else tmem_ld32x32b_x32_pair(t_o + c, t_o1 + c, o, o1);
#pragma unroll
            for (int e = 0; e < kEpi; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * c_self + __uint_as_float(o1[e]) * c_other);
          } else {
            if constexpr (kEpi == 64) tmem_ld32x32b_x64(t_o + c, o);
            else tmem_ld32x32b_x32(t_o + c, o);
#pragma unroll
            for (int e = 0; e < kEpi; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * c_self);
          }
          if constexpr (PARTIAL) {
            // fp32 partial rows: each warp stages its 32 rows as D/32 boxes of 32 rows x 32
            // columns (128-byte swizzled rows, 4 KB each), then stores them with TMA.
#pragma unroll
            for (int u = 0; u < kEpi / 4; ++u) {
              const int col = c + 4 * u;
              const uint32_t addr = part_box(col >> 5) + lane * 128 + ((((col & 31) >> 2) ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o[4 * u + 0]),
                           "r"(o[4 * u + 1]), "r"(o[4 * u + 2]), "r"(o[4 * u + 3])
                           : "memory");
            }
            continue;
          }
          if constexpr (L::kOneChunkStaging) {
            if (c > 0 && (c & 63) == 0) {
              // Store the previous 64-column chunk; its reads must finish before the staging
              // area is written again.
              fence_proxy_async_smem();
              __syncwarp();
              const int row0 = qt * kBM + wq * 32;
              if (lane == 0 && row0 < p.N) {
                tma_store_3d(&p.tm_o, ob + wq * 32 * 128, c - 64, row0, it.bh);
                bulk_commit_group();
                bulk_wait_group_read0();
              }
              __syncwarp();
            }
          }
          // 16-byte units (8 columns) of the 128-byte swizzled row of the 64-column chunk.
          const uint32_t row_base = ob + (L::kOneChunkStaging ? 0 : (c >> 6) * L::kChunkBytes) + r * 128;
#pragma unroll
          for (int u = 0; u < kEpi / 8; ++u) {
            const int unit = ((c & 63) >> 3) + u;
            const uint32_t addr = row_base + ((unit ^ (r & 7)) << 4);
            const uint32_t w0 = pack2<BF16>(__uint_as_float(o[8 * u + 0]), __uint_as_float(o[8 * u + 1]));
            const uint32_t w1 = pack2<BF16>(__uint_as_float(o[8 * u + 2]), __uint_as_float(o[8 * u + 3]));
            const uint32_t w2 = pack2<BF16>(__uint_as_float(o[8 * u + 4]), __uint_as_float(o[8 * u + 5]));
            const uint32_t w3 = pack2<BF16>(__uint_as_float(o[8 * u + 6]), __uint_as_float(o[8 * u + 7]));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                         : "memory");
          }
        }
        tc_fence_before();
        if (merge) mbar_arrive(bar(L::kO1Free));  // O1 and (m1, l1) consumed
        if (own_b) mbar_arrive(bar(L::kO1Self));  // O1 read for b's store
        if constexpr (PARTIAL) {
          if (row < p.N)
            p.lse_part[(static_cast<long long>(it.split) * p.BH + it.bh) * p.N + row] = (m_used + log2f(l_run)) * kLn2;
          fence_proxy_async_smem();
          __syncwarp();
          const int row0_warp = qt * kBM + wq * 32;
          if (lane == 0 && row0_warp < p.N) {
            for (int b = 0; b < D / 32; ++b)
              tma_store_3d(&p.tm_op, part_box(b), b * 32, row0_warp, it.split * p.BH + it.bh);
            bulk_commit_group();
          }
          continue;
        }
        if (p.lse != nullptr && row < p.N)
          p.lse[static_cast<long long>(it.bh) * p.N + row] = (m_used + log2f(l_run)) * kLn2;
        fence_proxy_async_smem();
        __syncwarp();
        const int row0_warp = qt * kBM + wq * 32;
        if (lane == 0 && row0_warp < p.N) {  // rows past N are clipped by the store; skip empty boxes
          if constexpr (L::kOneChunkStaging) {
            tma_store_3d(&p.tm_o, ob + wq * 32 * 128, D - 64, row0_warp, it.bh);
          } else {
            for (int c = 0; c < L::kChunks; ++c)
              tma_store_3d(&p.tm_o, ob + c * L::kChunkBytes + wq * 32 * 128, c * 64, row0_warp, it.bh);
          }
          bulk_commit_group();
        }
      }
      if (!ok) break;
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) grid_launch_dependents();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
