// attn_fwd.cuh -- warp-specialised causal prefill attention for GB300 (sm_103a).
//
// One persistent CTA per SM.  A work item is (batch b, query head h, query
// block qb) with two 128-row query tiles (rows 256*qb .. 256*qb+255); the two
// tiles share every K/V tile that TMA brings in.  Items run longest first
// (see decode_item for the chunked order of very large problems).  Problems
// with too few items to keep every SM busy run through the SPLIT kernels,
// where the longest items are split along the keys into pieces that run on
// different CTAs and are added up by the piece that finishes last (see
// decode_unit and split_arrive).  Roles (12 warps):
//   warps 0-3   softmax of query tile 0 (thread = row)
//   warps 4-7   softmax of query tile 1
//   warp  8     TMA producer: Q tiles once per item, K/V tiles through a ring
//   warp  9     QK issuer: S = Q_t K_j^T for (j, t) = (0,0), (0,1), (1,0), ...
//   warp  10    PV issuer: O_t += P_t V_j; owns tensor memory (BF16: each
//               P.V product is issued behind the tile's next S product)
//   warp  11    idle (completes the last warpgroup)
//
// Tensor memory (512 columns x 128 lanes of 32-bit words), FP8 paths:
//   S [0,128)  shared by both query tiles, handed over S0(j), S1(j), S0(j+1)...
//   P0 [128,160) SFA0 [160,164)  P1 [176,208) SFA1 [208,212)  SFB [216,221)
//   O0 [224,368)  O1 [368,512)   (144 columns: value dims + the row-sum column)
// BF16 path: S [0,128)  P0 [128,192)  P1 [192,256)  O0 [256,384)  O1 [384,512).
//
// A QK product is issued as soon as the softmax warpgroup that owned S has
// copied it into registers, so S for the next tile is computed while the
// softmax still works on the current one, and the P.V products are issued by
// their own warp whenever a P_t(j) is ready.  The softmax of each tile thus
// hides behind a whole period of tensor-core work (both tiles' QK and PV).
// Two issuing warps: the QK products wait on S hand-overs and the P.V
// products on P, and issuing four MMAs and a commit keeps a thread busy for
// about 275 clocks (more under contention), so one thread serving both waits
// would delay one product behind the other; its next wait would also stall
// until its own MMAs drain.  This replaces the "two-wave ping-pong"
// of the MI355X design ("Zyphra ZYFA: FP8 FlashAttention for AMD MI355X",
// "How does ZYFA work?"): asynchronous tcgen05 MMAs tracked by mbarriers
// provide the overlap.
//
// At the MLA shape the Lean-P paths write P in two 64-key halves, and the P.V
// warp issues each product's first two K-steps as soon as the first half is in
// tensor memory (Cfg::kPHalves).  An item ends with its epilogue in the
// softmax warps: out = dv * O / l, O read with one wait and released before
// the output is written; the Lean-P path writes bf16 rows into a 4 KB
// shared-memory slot per warp and stores them with TMA (Cfg::kEpiTma), so that
// the next item's first S product does not wait for scattered row stores.
//
// Probability policies (softmax warpgroups):
//   kLeanP     one saturating multiply-add per probability rounded toward
//              minus infinity, whose value floored to 1/128 is the e4m3 code,
//              and packed floors that gather four codes per word (see
//              leanp_codes4; "Lean P: one multiply-add instead of an
//              exponential"); a
//              power-of-two scale per 64-key block enters the P.V MMA as a
//              UE8M0 block-scale factor, and the P.V product runs against
//              [V | ones] so that column 128 of O accumulates the sum of the
//              rounded, scaled probabilities ("Per-block scaling and a rounded
//              row sum").
//   kExactFp8  p = 2^(x - m) on the MUFU, rounded to e4m3, unrounded row sum.
//   kBf16      as kExactFp8 with bf16 operands and probabilities.
//   kLeanPA3   kLeanP with the code grid anchored at the running row maximum
//              (the key holding it gets exactly the code of 2^T) instead of at
//              integer log2 values; O is rescaled exactly whenever the maximum
//              grows.
//   kBlockExact  diagnostic: the block exponents, UE8M0 factors and rounded
//              row sum of kLeanP, but each probability is 2^(x/8 - e + T) from
//              the MUFU rounded to the nearest e4m3 instead of the Lean-P
//              code, so that it differs from kLeanP in the code step alone.
#pragma once

#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace fa8 {

// Optional role timeline (debug builds with -DFA8_TIMELINE): clock64 stamps of
// CTA 0, written to fa8_timeline.  Roles 0-3: the first item, one row of
// stamps per key tile.  Roles 4-5: one row per item (round) of CTA 0, the
// events at the items' boundaries.
#ifdef FA8_TIMELINE
__device__ unsigned long long fa8_timeline[6][64][8];
#define FA8_TL(role, j, k)                                                    \
  do {                                                                        \
    if (blockIdx.x == 0 && (j) < 64) fa8_timeline[role][j][k] = clock64();    \
  } while (0)
#else
#define FA8_TL(role, j, k) \
  do {                     \
  } while (0)
#endif

enum Variant : int { kLeanP = 0, kExactFp8 = 1, kBf16 = 2, kBlockExact = 3, kLeanPA3 = 4 };

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kDV = 128;  // value head dim
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kQkWarp = 9;
constexpr int kPvWarp = 10;  // also allocates tensor memory

// Lean-P constants.  T = 7 headroom binades: the largest probability of each
// 64-key block gets a code in [C-8, C], C = 8*(7+T) = 112 (the code of 2^T).
constexpr int kLeanT = 7;
constexpr float kLeanC = 112.0f;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: floats in [2^23, 2^24) have unit spacing
// A row's reference binade is only raised when a block exponent exceeds it
// by more than this many binades (all rescales are exact powers of two).
constexpr float kLazyBinades = 8.0f;
// Running-maximum anchoring (kLeanPA3): the code of a key is
// floor(8*lam*(s - m) + 8k + C + eps), eps = 2^-6, so the key at the running
// maximum m gets exactly C, the code of 2^T.
constexpr float kA3Bias = kLeanC + 1.0f / 64.0f;

template <int V, int DQK>
struct Cfg {
  static constexpr bool kFp8 = V != kBf16;
  // per-64-key power-of-two block scale and the rounded row sum (O column 128)
  static constexpr bool kBlockScaled = V == kLeanP || V == kBlockExact || V == kLeanPA3;
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = DQK * kElem;             // bytes of one Q/K row
  static constexpr int kFullPanels = kRowBytes / 128;       // 128-byte swizzled panels
  static constexpr int kTailBytes = kRowBytes % 128;        // 0 or 64 (MLA shape)
  static constexpr int kPanelBytes = 128 * 128;             // 128 rows x 128 bytes
  static constexpr int kTailPanelBytes = 128 * kTailBytes;  // 128 rows x 64 bytes
  static constexpr int kQkTileBytes = kFullPanels * kPanelBytes + kTailPanelBytes;
  static constexpr int kVTileBytes = kBN * kDV * kElem;
  static constexpr int kVPanels = kDV * kElem / 128;
  static constexpr int kStages = kFp8 ? (DQK == 128 ? 4 : 3) : 2;
  // Q buffers.  With two (FP8 at head dim 128 has the shared memory for them)
  // the next item's Q tiles load while the current item runs; measured against
  // one buffer in one session that was 2-5% slower from 2K to 16K keys and on
  // the sink and GQA workloads, and 1.6% faster at 32K, so one is used.
  static constexpr int kQBufs = 1;
  static constexpr int kQBufBytes = 2 * kQkTileBytes;  // both query tiles of an item
  static constexpr int kSmemQ = 0;
  static constexpr int kSmemK = kQBufs * kQBufBytes;
  static constexpr int kSmemV = kSmemK + kStages * kQkTileBytes;
  // Lean-P: 128 keys x 128 bytes of e4m3 1.0, the second N-atom of the P.V
  // B operand, so that O's column 128 accumulates the rounded row sum
  static constexpr int kOnesBytes = kBlockScaled ? 128 * 128 : 0;
  static constexpr int kSmemOnes = kSmemV + kStages * kVTileBytes;
  // bf16 output through TMA stores: one 4 KB slot per softmax warp, 32 rows x
  // 64 columns in the 128-byte swizzle, stored in two halves, so that the
  // softmax warps do not wait for the scattered 16-byte row stores of the
  // BSHD layout at an item's end.  Measured against direct stores in one
  // session: Lean-P 2-8% faster from 2K to 8K keys and level at 16K-32K; the
  // other paths' softmax code compiled slower with it (the ablation by 13%),
  // so they keep direct stores.
  static constexpr bool kEpiTma = V == kLeanP;
  static constexpr int kOutSlotBytes = 32 * 128;
  static constexpr int kSmemOut = kSmemOnes + kOnesBytes;  // a multiple of 1024
  static constexpr int kSmemBytes = kSmemOut + (kEpiTma ? 8 * kOutSlotBytes : 0);
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
  static constexpr int kQkSteps = kRowBytes / 32;       // one MMA per 32 bytes of K
  static constexpr int kPvSteps = kFp8 ? 4 : 8;         // 128 keys / (32 fp8 or 16 bf16)
  static constexpr int kPCols = kFp8 ? 32 : 64;         // TMEM columns of P per tile
  static constexpr int kPvN = kBlockScaled ? 144 : 128;  // P.V N (with the ones column)
  // BF16: P.V of key tile j waits until the tile's S product of key tile j+1
  // is issued (see pv_loop).  Measured on the FP8 paths, the same order was
  // slower: there the P.V warp's issue-and-drain then delays P.V past the
  // point where the softmax needs it.
  static constexpr bool kOrderPv = !kFp8;
  // P written and announced in two 64-key halves, each P.V product issued as
  // two pairs of K-steps, the first as soon as its half is in tensor memory.
  // Measured against whole P in one session: 1.2% (integer binades) and 2.1%
  // (running-maximum anchor) faster at the MLA shape, where the S product is
  // six MMAs, but 1-3% slower at head dim 128 and slower on the exact paths.
  static constexpr bool kPHalves = DQK == 192 && (V == kLeanP || V == kLeanPA3);
  // epilogue: all of O_t read with one wait and O_t released before the
  // output stores (FP8 paths; the BF16 softmax, short of registers already,
  // measured 12% slower with the 128-column read)
  static constexpr bool kEarlyOFree = kFp8;
  // the softmax works out each item's coordinates and loads its descales
  // before the previous item's epilogue.  Measured against the plain order in
  // two sessions: Lean-P at head dim 128 3% faster at 32K and level from 2K to
  // 16K; 1.5% slower at the MLA shape, and the other paths' softmax compiled
  // slower with it (the ablation by 13%).
  static constexpr bool kPrefetchItem = V == kLeanP && DQK == 128;
  // tensor-memory columns
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColP0 = 128, kColP1 = kFp8 ? 176 : 192;
  static constexpr uint32_t kColSfb = 216;  // FP8 only
  static constexpr uint32_t kColO0 = kFp8 ? 224 : 256, kColO1 = kFp8 ? 368 : 384;
  static_assert(kTailBytes == 0 || kTailBytes == 64, "row bytes must be 128*n or 128*n+64");
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");
  static_assert(kSmemOut % 1024 == 0, "128-byte swizzled slots need 1024-byte alignment");
};

struct KParams {
  int B, Hq, Hkv, S;
  int group;         // Hq / Hkv
  int n_qblocks;     // ceil(S / 256)
  int n_kv_tiles;    // ceil(S / 128)
  int n_items;       // B * Hq * n_qblocks
  int n_units;       // work units: n_items, plus split_ns - 1 per split item
  const float* dq;   // device descales (FP8 only)
  const float* dk;
  const float* dv;
  float scale;       // softmax scale
  void* out;
  int out_f32;
  int* status;       // optional device status word
  int flags;
  unsigned long long wait_limit_ns;
  int chunk_q;         // query-head units (b, h) per item chunk, a multiple of Hq / Hkv
  int causal;          // 1: keys j <= i; 0: all S keys
  int descale_per_bkv; // descales hold one value per (batch, kv head) instead of one
  float* lse;          // optional [B, Hq, S] natural-log row sums (nullptr: none)
  // Split schedule (SPLIT kernels only): the items of query block >= split_qb,
  // the first n_split_items of the plain order, run as split_ns pieces each.
  int split_qb, split_ns, n_split_items;
  unsigned char* ws;             // workspace: counters, then partial results
  unsigned long long epoch;      // this call's tag in the counters (< 2^61)
};

// Split workspace layout: one 64-bit counter per (split item, query tile),
// padded to 256 bytes, then one slot per (split item, piece, query tile) of
// kSplitSlotFloats floats: O as [32 column quads][128 rows] float4, then the
// row sums l[128] and the reference binades ref[128].
constexpr int kSplitSlotFloats = 128 * 128 + 2 * 128;
__host__ __device__ constexpr size_t split_cnt_bytes(int n_split_items) {
  return ((size_t)n_split_items * 16 + 255) / 256 * 256;
}

struct Maps {
  CUtensorMap q128, k128, v;  // 128-byte panels (SW128)
  CUtensorMap q64, k64;       // 64-byte tail panel of the MLA shape (SW64)
  CUtensorMap o64;            // bf16 output, boxes of 64 columns x 32 rows (SW128)
};

// Items are visited longest first (query block descending); CTA c takes the
// c-th item of each round of gridDim.x items, alternating direction every
// round, so that every CTA gets a similar share of causal work.
__device__ __forceinline__ int item_at(int round, int n_items) {
  const int G = gridDim.x;
  const int pos = round * G + ((round & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return pos < n_items ? pos : -1;
}

// Item order: the query-head units q = b*Hq + h are split into chunks of
// chunk_q consecutive units (whole kv heads); chunks run one after another,
// and inside a chunk the query blocks run longest first with the units as the
// fast index.  One chunk (chunk_q = B*Hq) is the plain longest-first order.
// Smaller chunks keep the CTAs in flight on few kv heads, so that their K and
// V tiles are shared in L2 when all heads' K and V would not fit there.
__device__ __forceinline__ void decode_item(const KParams& p, int idx, int& b, int& h, int& qb) {
  const int units = p.B * p.Hq;
  const int per_chunk = p.chunk_q * p.n_qblocks;
  const int c = idx / per_chunk;
  const int q0 = c * p.chunk_q;
  const int cq = units - q0 < p.chunk_q ? units - q0 : p.chunk_q;
  const int li = idx - c * per_chunk;
  qb = p.n_qblocks - 1 - li / cq;
  const int q = q0 + li % cq;
  b = q / p.Hq;
  h = q % p.Hq;
}

// Number of key tiles query tile t of block qb needs (keys < min(S, last row + 1)).
__device__ __forceinline__ int kv_tiles_for(const KParams& p, int qb, int t) {
  const int need = 2 * qb + t + 1;
  return p.causal && need < p.n_kv_tiles ? need : p.n_kv_tiles;
}

// A work unit: a whole item, or (SPLIT kernels) one piece of a split item,
// which covers key tiles [j0, end_t) of query tile t.
struct Unit {
  int u;          // unit index
  int b, h, qb;
  int j0, end0, end1;
  int piece, ns;  // piece of ns (ns = 1: the whole item)
  int sidx;       // split item index: its counters and partial results
};

// Unit u: with a split schedule the first n_split_items * split_ns units are
// the pieces of the split items (consecutive pieces of one item), the rest the
// other items in the plain order.  Piece s covers key tiles
// [s*n/ns, (s+1)*n/ns) of the item's n; the schedule splits only items with
// n >= 2*ns, so every piece gives both query tiles at least one key tile.
template <bool SPLIT>
__device__ __forceinline__ void decode_unit(const KParams& p, int u, Unit& w) {
  int idx = u;
  w.u = u;
  w.piece = 0;
  w.ns = 1;
  w.sidx = 0;
  if constexpr (SPLIT) {
    const int n_split_units = p.n_split_items * p.split_ns;
    if (u < n_split_units) {
      w.sidx = u / p.split_ns;
      w.piece = u - w.sidx * p.split_ns;
      w.ns = p.split_ns;
      idx = w.sidx;
    } else {
      idx = u - n_split_units + p.n_split_items;
    }
  }
  decode_item(p, idx, w.b, w.h, w.qb);
  w.j0 = 0;
  w.end0 = kv_tiles_for(p, w.qb, 0);
  w.end1 = kv_tiles_for(p, w.qb, 1);
  if constexpr (SPLIT) {
    if (w.ns > 1) {
      const int n = w.end1;
      w.j0 = w.piece * n / w.ns;
      w.end1 = (w.piece + 1) * n / w.ns;
      w.end0 = w.end0 < w.end1 ? w.end0 : w.end1;
    }
  }
}

// The arrival of one finished piece of split item sidx, query tile t, after
// its partial result is in the workspace (and fenced): true for the piece
// that arrives last.  The counter holds (epoch << 3) + pieces arrived; a
// value with another epoch (an earlier call, or memory never used) counts as
// zero, so the workspace needs no clearing between calls.  The last piece
// sets the counter back to zero: every piece of this call has arrived, and a
// replay of the same launch from a CUDA graph, which repeats its epoch, then
// starts from zero too.
__device__ __forceinline__ bool split_arrive(const KParams& p, int sidx, int ns, int t,
                                             volatile int* ab) {
  unsigned long long* cnt = reinterpret_cast<unsigned long long*>(p.ws) + (size_t)sidx * 2 + t;
  unsigned long long old = atomicAdd(cnt, 0ull);
  for (int it = 0;; ++it) {
    const unsigned long long nw = (old >> 3) == p.epoch ? old + 1 : (p.epoch << 3) + 1;
    const unsigned long long prev = atomicCAS(cnt, old, nw);
    if (prev == old) break;
    old = prev;
    if (it > 64) {  // only the other pieces move the counter: a few retries at most
      *ab = 1;
      return false;
    }
  }
  const unsigned long long before = (old >> 3) == p.epoch ? (old & 7ull) : 0ull;
  const bool last = before == (unsigned long long)(ns - 1);
  if (last) atomicExch(cnt, 0ull);
  return last;
}

struct __align__(8) Barriers {
  uint64_t q_full[2], q_empty[2];  // per Q buffer
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2];     // S holds S_t(j) (QK commit)
  uint64_t s_drained[2];  // softmax t has copied S into registers
  uint64_t p_full[2];     // softmax t has written P_t(j)
  uint64_t p_half[2];     // softmax t has written the first 64 keys of P_t(j) (FP8)
  uint64_t o_done[2];     // PV_t(j) complete (PV commit)
  uint64_t qk_go[2][4];   // S product n of tile t issued: qk_go[t][n % 4] (BF16)
  uint64_t o_free[2];     // softmax t has read O_t in its epilogue
  uint64_t drain[2];      // teardown: all MMAs of the QK / PV warp complete
  uint64_t split_sync[2]; // SPLIT: the 128 threads of softmax t (a bounded group barrier)
  uint32_t tmem_base;
  int abort_flag;
  int split_last[2];      // SPLIT: this query tile's piece arrived last
};

// --------------------------------------------------------------------------
// Producer warp: TMA loads.
// --------------------------------------------------------------------------
template <int V, int DQK>
__device__ __forceinline__ void load_qk_tile(uint8_t* dst, const Maps& m, bool is_q,
                                             uint64_t* bar, int head, int row, int b) {
  using C = Cfg<V, DQK>;
  const CUtensorMap* full = is_q ? &m.q128 : &m.k128;
#pragma unroll
  for (int pnl = 0; pnl < C::kFullPanels; ++pnl)
    tma_load_4d(dst + pnl * C::kPanelBytes, full, bar, pnl * (128 / C::kElem), head, row, b);
  if constexpr (C::kTailBytes) {
    const CUtensorMap* tail = is_q ? &m.q64 : &m.k64;
    tma_load_4d(dst + C::kFullPanels * C::kPanelBytes, tail, bar,
                C::kFullPanels * (128 / C::kElem), head, row, b);
  }
}

template <int V, int DQK, bool SPLIT>
__device__ void producer_loop(const KParams& p, const Maps& m, uint8_t* smem, Barriers& bars) {
  using C = Cfg<V, DQK>;
  if (!elect_one()) return;
  if (p.flags & 1) return;  // test hook: issue nothing, every consumer wait expires
  prefetch_tmap(&m.q128);
  prefetch_tmap(&m.k128);
  prefetch_tmap(&m.v);
  volatile int* ab = &bars.abort_flag;
  uint32_t kv_it = 0, q_it = 0, nk = 0, nv = 0;
  for (int round = 0;; ++round) {
    const int u = item_at(round, p.n_units);
    if (u < 0) break;
    Unit w;
    decode_unit<SPLIT>(p, u, w);
    const int b = w.b, h = w.h, qb = w.qb;
    const int g = h / p.group;
    const uint32_t qbuf = q_it % C::kQBufs, qph = (q_it / C::kQBufs) & 1;
    if (!mbar_wait(&bars.q_empty[qbuf], qph ^ 1, ab, p.wait_limit_ns)) break;
    uint8_t* qdst = smem + C::kSmemQ + qbuf * C::kQBufBytes;
    FA8_TL(4, round, 0);
    mbar_arrive_expect_tx(&bars.q_full[qbuf], 2 * C::kQkTileBytes);
    load_qk_tile<V, DQK>(qdst, m, true, &bars.q_full[qbuf], h, qb * 256, b);
    load_qk_tile<V, DQK>(qdst + C::kQkTileBytes, m, true, &bars.q_full[qbuf], h, qb * 256 + 128,
                         b);
    ++q_it;
    const int nkv = w.end1;
    for (int j = w.j0; j < nkv; ++j, ++kv_it) {
      const uint32_t st = kv_it % C::kStages, ph = (kv_it / C::kStages) & 1;
      if (!mbar_wait(&bars.k_empty[st], ph ^ 1, ab, p.wait_limit_ns)) break;
      mbar_arrive_expect_tx(&bars.k_full[st], C::kQkTileBytes);
      load_qk_tile<V, DQK>(smem + C::kSmemK + st * C::kQkTileBytes, m, false, &bars.k_full[st], g,
                           j * kBN, b);
      if (j == w.j0) FA8_TL(4, round, 1);
      ++nk;
      if (!mbar_wait(&bars.v_empty[st], ph ^ 1, ab, p.wait_limit_ns)) break;
      ++nv;
      mbar_arrive_expect_tx(&bars.v_full[st], C::kVTileBytes);
#pragma unroll
      for (int pnl = 0; pnl < C::kVPanels; ++pnl)
        tma_load_4d(smem + C::kSmemV + st * C::kVTileBytes + pnl * C::kPanelBytes, &m.v,
                    &bars.v_full[st], pnl * (128 / C::kElem), g, j * kBN, b);
    }
    if (*ab) break;
  }
  // Before the CTA may exit, every copy this thread started must have landed:
  // after an abort, and also after a normal end, since a wait in another role
  // may still run out of time while the last loads are in flight.  Only the
  // last kStages loads of K and of V, and the last kQBufs loads of Q, can be
  // in flight (a buffer is reloaded only after its consumer has waited for
  // the previous load).
  // A drain that runs out of time is reported like any other expired wait.
  constexpr uint64_t kDrainNs = 50000000ull;
  volatile int gave_up = 0;
  bool ok = true;
  for (uint32_t i = nk > (uint32_t)C::kStages ? nk - C::kStages : 0; i < nk; ++i)
    ok &= mbar_wait(&bars.k_full[i % C::kStages], (i / C::kStages) & 1, &gave_up, kDrainNs);
  for (uint32_t i = nv > (uint32_t)C::kStages ? nv - C::kStages : 0; i < nv; ++i)
    ok &= mbar_wait(&bars.v_full[i % C::kStages], (i / C::kStages) & 1, &gave_up, kDrainNs);
  for (uint32_t i = q_it > (uint32_t)C::kQBufs ? q_it - C::kQBufs : 0; i < q_it; ++i)
    ok &= mbar_wait(&bars.q_full[i % C::kQBufs], (i / C::kQBufs) & 1, &gave_up, kDrainNs);
  if (!ok) *ab = 1;
}

// --------------------------------------------------------------------------
// MMA issue.
// --------------------------------------------------------------------------
template <int V, int DQK>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t smem_base, uint32_t q_buf_off,
                                         int t, uint32_t k_off) {
  using C = Cfg<V, DQK>;
  constexpr uint32_t idesc = idesc_f32acc(128, 128, C::kFp8 ? 0 : 1, C::kFp8 ? 0 : 1, 0, 0);
  const uint32_t q_off = q_buf_off + t * C::kQkTileBytes;
#pragma unroll
  for (int k = 0; k < C::kQkSteps; ++k) {
    const int byte = 32 * k;
    const int pnl = byte / 128;
    uint64_t a, bdesc;
    if (pnl < C::kFullPanels) {
      const uint32_t o = pnl * C::kPanelBytes + (byte % 128);
      a = smem_desc(smem_base + q_off + o, 16, 1024, kSwizzle128B);
      bdesc = smem_desc(smem_base + k_off + o, 16, 1024, kSwizzle128B);
    } else {
      const uint32_t o = C::kFullPanels * C::kPanelBytes + (byte % 128);
      a = smem_desc(smem_base + q_off + o, 16, 512, 4);
      bdesc = smem_desc(smem_base + k_off + o, 16, 512, 4);
    }
    if constexpr (C::kFp8)
      mma_f8_ss(tmem + C::kColS, a, bdesc, idesc, k > 0);
    else
      mma_f16_ss(tmem + C::kColS, a, bdesc, idesc, k > 0);
  }
}

// K-steps K0 .. K1-1 of O_t (+)= P_t V (32 keys per FP8 step, 16 per BF16 step).
template <int V, int DQK, int K0, int K1>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint32_t smem_base, int t, uint32_t v_off,
                                         bool accumulate) {
  using C = Cfg<V, DQK>;
  const uint32_t d = tmem + (t ? C::kColO1 : C::kColO0);
  const uint32_t a = tmem + (t ? C::kColP1 : C::kColP0);
  if constexpr (C::kFp8) {
    // SFA of P_t at a + 32 (+ lane quadrant, the MMA's read pattern), byte =
    // K-step; SFB (all 1.0) at kColSfb.  Lean-P: B = [V | ones], the ones atom
    // at LBO after the V stage; N = 128 otherwise.
    const uint32_t lbo = C::kOnesBytes ? (uint32_t)(C::kSmemOnes - (int)v_off) : 1024u;
#pragma unroll
    for (int k = K0; k < K1; ++k) {
      const uint64_t bdesc = smem_desc(smem_base + v_off + 4096 * k, lbo, 1024, kSwizzle128B);
      mma_mx8_ts(d, a + 8 * k, bdesc, idesc_mx(128, C::kPvN, 0, 0, 0, 1, k, k), a + 32,
                 tmem + C::kColSfb, accumulate || k > 0);
    }
  } else {
    constexpr uint32_t idesc = idesc_f32acc(128, 128, 1, 1, 0, 1);
#pragma unroll
    for (int k = K0; k < K1; ++k) {
      const uint64_t bdesc =
          smem_desc(smem_base + v_off + 2048 * k, C::kPanelBytes, 1024, kSwizzle128B);
      mma_f16_ts(d, a + 8 * k, bdesc, idesc, accumulate || k > 0);
    }
  }
}

// QK warp: S = Q_t K_j^T in the order S0(0), S1(0), S0(1), S1(1), ... (tile 0
// skips key tiles past its diagonal).  Each product waits until the previous
// owner of S has copied it out.
template <int V, int DQK, bool SPLIT>
__device__ void qk_loop(const KParams& p, uint32_t smem_base, Barriers& bars, uint32_t tmem) {
  using C = Cfg<V, DQK>;
  if (lane_id() != 0) return;
  volatile int* ab = &bars.abort_flag;
  const uint64_t lim = p.wait_limit_ns;
  uint32_t kv_it = 0, q_it = 0;
  uint32_t issued[2] = {0, 0};  // S products issued per tile
  int last = -1;                // tile of the previous S product
  for (int round = 0;; ++round) {
    const int u = item_at(round, p.n_units);
    if (u < 0) break;
    Unit w;
    decode_unit<SPLIT>(p, u, w);
    const int nk0 = w.end0, nkv = w.end1;
    const uint32_t qbuf = q_it % C::kQBufs;
    const uint32_t q_buf_off = C::kSmemQ + qbuf * C::kQBufBytes;
    if (!mbar_wait(&bars.q_full[qbuf], (q_it / C::kQBufs) & 1, ab, lim)) return;
    FA8_TL(4, round, 2);
    ++q_it;
    for (int j = w.j0; j < nkv; ++j, ++kv_it) {
      const uint32_t st = kv_it % C::kStages, ph = (kv_it / C::kStages) & 1;
      if (!mbar_wait(&bars.k_full[st], ph, ab, lim)) return;
      for (int t = 0; t < 2; ++t) {
        if (j >= (t ? nkv : nk0)) continue;
        const bool stamp = round == 0;
        if (stamp) FA8_TL(2 + t, j, 3);
        if (last >= 0 &&
            !mbar_wait(&bars.s_drained[last], (issued[last] - 1) & 1, ab, lim))
          return;
        if (stamp) FA8_TL(2 + t, j, 4);
        tc_fence_after();
        issue_qk<V, DQK>(tmem, smem_base, q_buf_off, t, C::kSmemK + st * C::kQkTileBytes);
        // the P.V warp may now queue this tile's previous P.V product behind it
        if constexpr (C::kOrderPv) mbar_arrive(&bars.qk_go[t][issued[t] & 3]);
        tc_commit(&bars.s_full[t]);
        if (stamp) FA8_TL(2 + t, j, 5);
        if (j == w.j0 && t == 0) FA8_TL(4, round, 3);
        ++issued[t];
        last = t;
      }
      tc_commit(&bars.k_empty[st]);
    }
    FA8_TL(4, round, 4);
    tc_commit(&bars.q_empty[qbuf]);
  }
}

// PV warp: O_t += P_t V_j as soon as P_t(j) is written.  With kOrderPv (BF16)
// it also waits until S_t(j+1) has been issued, unless j is the tile's last key
// tile: the tensor pipe runs products in issue order, so the S product, which
// the other tile's softmax is about to wait for, does not queue behind a P.V
// product that became ready at the same moment.  The QK warp arrives on
// qk_go[t][n % 4] after issuing S product n of tile t, counted over all items,
// and this warp consumes every arrival in order (at a tile's last key tile up
// to S_t(j) itself, already issued).  No barrier can run two phases ahead of
// this warp: the next arrival on the barrier of n is n + 4, and S_t(n+4) is
// issued only after the softmax has written P_t at a key tile two or more past
// the P.V product that consumes n, which waits for that P.V product.  (With
// two barriers this fails at an item's start, where P_t(0) is written without
// waiting for any P.V product.)
template <int V, int DQK, bool SPLIT>
__device__ void pv_loop(const KParams& p, uint32_t smem_base, Barriers& bars, uint32_t tmem) {
  using C = Cfg<V, DQK>;
  if (lane_id() != 0) return;
  volatile int* ab = &bars.abort_flag;
  const uint64_t lim = p.wait_limit_ns;
  uint32_t kv_it = 0, p_cnt[2] = {0, 0}, items = 0;
  uint32_t qk_base[2] = {0, 0};  // S products of each tile in earlier items
  uint32_t go_seen[2] = {0, 0};  // qk_go arrivals consumed per tile
  for (int round = 0;; ++round) {
    const int u = item_at(round, p.n_units);
    if (u < 0) break;
    Unit w;
    decode_unit<SPLIT>(p, u, w);
    const int nk0 = w.end0, nkv = w.end1, j0 = w.j0;
    for (int j = j0; j < nkv; ++j, ++kv_it) {
      const uint32_t st = kv_it % C::kStages, ph = (kv_it / C::kStages) & 1;
      const bool stamp = round == 0;
      if (!mbar_wait(&bars.v_full[st], ph, ab, lim)) return;
      for (int t = 0; t < 2; ++t) {
        if (j >= (t ? nkv : nk0)) continue;
        if (stamp) FA8_TL(2 + t, j, 0);
        if (!mbar_wait(C::kPHalves ? &bars.p_half[t] : &bars.p_full[t], p_cnt[t] & 1, ab, lim))
          return;
        if (j == j0) {
          // the previous unit's epilogue must have read O_t
          if (!mbar_wait(&bars.o_free[t], (items & 1) ^ 1, ab, lim)) return;
        }
        if constexpr (C::kOrderPv) {
          const int nk = t ? nkv : nk0;
          const uint32_t upto = qk_base[t] + (j + 1 < nk ? j + 1 : j) - j0;
          for (; go_seen[t] <= upto; ++go_seen[t])
            if (!mbar_wait(&bars.qk_go[t][go_seen[t] & 3], (go_seen[t] >> 2) & 1, ab, lim))
              return;
        }
        if (stamp) FA8_TL(2 + t, j, 1);
        tc_fence_after();
        const uint32_t v_off = C::kSmemV + st * C::kVTileBytes;
        if constexpr (C::kPHalves) {
          issue_pv<V, DQK, 0, 2>(tmem, smem_base, t, v_off, j > j0);
          if (!mbar_wait(&bars.p_full[t], p_cnt[t] & 1, ab, lim)) return;
          tc_fence_after();
          issue_pv<V, DQK, 2, 4>(tmem, smem_base, t, v_off, true);
        } else {
          issue_pv<V, DQK, 0, C::kPvSteps>(tmem, smem_base, t, v_off, j > j0);
        }
        ++p_cnt[t];
        tc_commit(&bars.o_done[t]);
        if (stamp) FA8_TL(2 + t, j, 2);
        if (j == j0 && t == 0) FA8_TL(4, round, 5);
      }
      tc_commit(&bars.v_empty[st]);
    }
    FA8_TL(4, round, 6);
    qk_base[0] += nk0 - j0;
    qk_base[1] += nkv - j0;
    ++items;
  }
}

// --------------------------------------------------------------------------
// Softmax warpgroups.
// --------------------------------------------------------------------------
// Four Lean-P codes c_i = clamp(floor(x_i), 0, .) with x_i = s_i*lam8 + C - 8e,
// one per byte of the result (little-endian, s0 in the low byte).
// `A` = lam8/128 and `b` = (C - 8e)/128 are exact power-of-two scalings, so
// t_i = RD(x_i/128) clamped to [0, 1] satisfies floor(128 t_i) = floor(x_i) for
// x_i >= 0 (floor(x_i)/128 is a float no larger than x_i/128) and 0 below.
// The floors are then taken two lanes at a time by rounding down into ranges
// of fixed spacing: 2^31 (spacing 256) turns t into 2^31 + 256 c, adding
// 1.5*2^23 - 2^31 (exact) rebases it to 1.5*2^23 + 256 c, and a last rounded-down
// multiply-add of the partner lane (spacing 1) gives 1.5*2^23 + c_lo + 256 c_hi,
// whose two low bytes are the pair of codes.  Everything but the byte
// shuffle runs on the FMA pipe.
struct LeanPConsts {
  uint64_t k32768, base_hi, rebase, k128;
};
__device__ __forceinline__ LeanPConsts leanp_consts() {
  return {f32x2_pack(32768.0f, 32768.0f), f32x2_pack(2147483648.0f, 2147483648.0f),
          f32x2_pack(kMagic - 2147483648.0f, kMagic - 2147483648.0f), f32x2_pack(128.0f, 128.0f)};
}
__device__ __forceinline__ uint32_t leanp_codes4(float s0, float s1, float s2, float s3, float A,
                                                 float b, const LeanPConsts& k) {
  const float t0 = fma_rm_sat(s0, A, b), t1 = fma_rm_sat(s1, A, b);
  const float t2 = fma_rm_sat(s2, A, b), t3 = fma_rm_sat(s3, A, b);
  uint64_t z = fma_rm_f32x2(f32x2_pack(t1, t3), k.k32768, k.base_hi);  // 2^31 + 256 c_{1,3}
  z = add_f32x2(z, k.rebase);                                           // M + 256 c_{1,3}
  const uint64_t y = fma_rm_f32x2(f32x2_pack(t0, t2), k.k128, z);       // M + c_{0,2} + 256 c_{1,3}
  uint32_t y01, y23;
  f32x2_unpack(y, y01, y23);
  return prmt(y01, y23, 0x5410);
}

// Largest of the 64 fp32 values s[o .. o+63] (bit patterns): 32 three-input
// maxima (ALU pipe), four independent chains of 15 elements, then the last
// four elements folded into the combination.
__device__ __forceinline__ float block_max64(const uint32_t (&s)[128], int o) {
  auto f = [&](int i) { return __uint_as_float(s[o + i]); };
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmax3(f(i), f(4 + i), f(8 + i));  // elements 0 .. 11
#pragma unroll
  for (int c = 12; c < 60; c += 8) {  // elements 12 .. 59
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = fmax3(m[i], f(c + i), f(c + 4 + i));
  }
  const float a = fmax3(m[0], m[1], f(60)), bb = fmax3(m[2], m[3], f(61));
  return fmax3(a, bb, fmaxf(f(62), f(63)));
}

__device__ __forceinline__ float pow2i(int e) {  // exact 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

// Every lane waits; the warp proceeds only if all lanes saw the phase
// complete, so warp-collective tcgen05 instructions never run with part of
// the warp gone on the abort path.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* ab,
                                          uint64_t lim) {
  const bool ok = mbar_wait(bar, parity, ab, lim);
  return __all_sync(0xffffffffu, ok);
}

template <int V, int DQK, bool SPLIT>
__device__ void softmax_loop(const KParams& p, const Maps& maps, uint8_t* smem, Barriers& bars,
                             uint32_t tmem, int t) {
  using C = Cfg<V, DQK>;
  volatile int* ab = &bars.abort_flag;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t quad = warp_id() & 3;
  const int r = (int)(quad * 32 + lane_id());  // row within the query tile
  const uint32_t lane_base = (quad * 32) << 16;
  const uint32_t s_col = tmem + lane_base + C::kColS;
  const uint32_t p_col = tmem + lane_base + (t ? C::kColP1 : C::kColP0);
  const uint32_t o_col = tmem + lane_base + (t ? C::kColO1 : C::kColO0);
  const float log2e = 1.4426950408889634f;
  const LeanPConsts kc = leanp_consts();
  uint32_t s_cnt = 0, o_cnt = 0;
  uint32_t sync_cnt = 0;  // SPLIT: phases of split_sync[t] passed
  // The next item's coordinates and descales, worked out one item ahead
  // (kPrefetchItem): issued before the previous item's epilogue, the index
  // divisions and the descales' global-memory latency are not between that
  // epilogue and this item's first S hand-over.
  Unit nw{};
  bool nvalid = false;
  float dqk_next = 1.0f, dvv_next = 1.0f;
  auto prefetch_item = [&](int round_) {
    const int u_ = item_at(round_, p.n_units);
    nvalid = u_ >= 0;
    if (!nvalid) return;
    decode_unit<SPLIT>(p, u_, nw);
    if constexpr (C::kFp8) {
      const int di = p.descale_per_bkv ? nw.b * p.Hkv + nw.h / p.group : 0;
      dqk_next = __ldg(p.dq + di) * __ldg(p.dk + di);
      dvv_next = __ldg(p.dv + di);
    }
  };
  if constexpr (C::kPrefetchItem) prefetch_item(0);

  for (int round = 0;; ++round) {
    Unit w;
    float dqk = 1.0f, dvv = 1.0f;  // descales of this (batch, kv head)
    if constexpr (C::kPrefetchItem) {
      if (!nvalid) break;
      w = nw;
      dqk = dqk_next, dvv = dvv_next;
    } else {
      const int u = item_at(round, p.n_units);
      if (u < 0) break;
      decode_unit<SPLIT>(p, u, w);
      if constexpr (C::kFp8) {
        const int di = p.descale_per_bkv ? w.b * p.Hkv + w.h / p.group : 0;
        dqk = __ldg(p.dq + di) * __ldg(p.dk + di);
        dvv = __ldg(p.dv + di);
      }
    }
    const int b = w.b, h = w.h, qb = w.qb;
    const int j0 = SPLIT ? w.j0 : 0;
    const int nk = SPLIT ? (t ? w.end1 : w.end0) : kv_tiles_for(p, qb, t);
    const float lam = log2e * p.scale * dqk;  // log2 units per unit of s
    const float lam8 = 8.0f * lam;            // Lean-P code units per unit of s
    const float lamc = lam8 * (1.0f / 128.0f);
    const int row = qb * 256 + t * 128 + r;
    float l = 0.0f;    // exact paths: row sum of the unrounded probabilities
    float ref = 0.0f;  // Lean-P: reference binade; exact paths: running max (log2 units)
    bool have_ref = false;
    const bool stamp = round == 0 && r == 0;
    for (int j = j0; j < nk; ++j) {
      if (stamp) FA8_TL(t, j, 0);
      if (!warp_wait(&bars.s_full[t], s_cnt & 1, ab, lim)) return;
      if (stamp) FA8_TL(t, j, 1);
      if (j == j0 && r == 0) FA8_TL(5, round, 4 * t);
      ++s_cnt;
      tc_fence_after();
      uint32_t s[128];
      {
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        uint32_t (&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[64]);
        uint32_t (&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[96]);
        tmem_ld32x2_wait(s_col, s_col + 32, s0, s1);
        tmem_ld32x2_wait(s_col + 64, s_col + 96, s2, s3);
      }
      // S is in registers: the QK warp may reuse it for the other tile
      tc_fence_before();
      mbar_arrive(&bars.s_drained[t]);
      if (stamp) FA8_TL(t, j, 2);
      const int key0 = j * kBN;
      // the last key this row sees: itself (causal) or the last one (S - 1)
      const int kmax = p.causal ? row : p.S - 1;
      if (key0 + kBN - 1 > kmax) {  // diagonal or ragged tile: mask the keys beyond
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (key0 + c > kmax) s[c] = __float_as_uint(-INFINITY);
      }
      bool rescale = false;
      float alpha = 1.0f;
      uint32_t pw[C::kPCols];
      uint32_t sfa = 0x7F7F7F7Fu;
      // per-tile constants of the code step: the bias of each 64-key block
      // (Lean-P paths), the exponent offset of each block (block-exact), or
      // minus the running maximum (exact paths)
      float cb0 = 0.0f, cb1 = 0.0f;
      float ls0 = 0.f, ls1 = 0.f;  // exact paths: row sum of the unrounded p
      if constexpr (V == kLeanPA3) {
        // Codes anchored at the running maximum m (raw-score units; lam > 0):
        // k = floor(lam*(m - block max)) and the bias (8k + C + eps - 8 lam m)/128
        // per 64-key block.  O and its row-sum column are rescaled by
        // 2^(lam*(m_old - m_new)) whenever m grows.
        const float m0 = block_max64(s, 0), m1 = block_max64(s, 64);
        const float mt = fmaxf(m0, m1);
        if (!have_ref) {
          ref = mt;
          have_ref = true;
        } else if (mt > ref) {
          alpha = ex2_approx((ref - mt) * lam);
          ref = mt;
          rescale = true;
        }
        const bool v0 = m0 > -INFINITY, v1 = m1 > -INFINITY;
        const float k0 = v0 ? floorf((ref - m0) * lam) : 0.0f;
        const float k1 = v1 ? floorf((ref - m1) * lam) : 0.0f;
        // UE8M0 scale 2^(-T-k): byte 127 - T - k, at least 0 (k >= 0)
        const int x0 = v0 ? (int)fmaxf(127.0f - kLeanT - k0, 0.0f) : 0;
        const int x1 = v1 ? (int)fmaxf(127.0f - kLeanT - k1, 0.0f) : 0;
        // a fully masked block has only -inf scores: code 0 whatever the bias
        cb0 = v0 ? fmaf(-lam8, ref, 8.0f * k0 + kA3Bias) * (1.0f / 128.0f) : 0.0f;
        cb1 = v1 ? fmaf(-lam8, ref, 8.0f * k1 + kA3Bias) * (1.0f / 128.0f) : 0.0f;
        sfa = (uint32_t)x0 | ((uint32_t)x0 << 8) | ((uint32_t)x1 << 16) | ((uint32_t)x1 << 24);
      } else if constexpr (C::kBlockScaled) {
        const float m0 = block_max64(s, 0), m1 = block_max64(s, 64);
        // block exponents e = ceil(lam*max): the block maximum lands in (2^(T-1), 2^T]
        const float e0 = ceilf(m0 * lam8 * 0.125f), e1 = ceilf(m1 * lam8 * 0.125f);
        const float emax = fmaxf(e0, e1);
        if (!have_ref) {
          ref = emax;
          have_ref = true;
        } else if (emax > ref + kLazyBinades) {
          const float d = ref - emax;
          alpha = d < -126.0f ? 0.0f : pow2i((int)d);
          ref = emax;
          rescale = true;
        }
        // UE8M0 scale of each block: 2^(e - T - ref), clamped to the format
        const bool v0 = e0 > -INFINITY, v1 = e1 > -INFINITY;
        const int x0 = v0 ? max(min((int)(e0 - ref) - kLeanT + 127, 254), 0) : 0;
        const int x1 = v1 ? max(min((int)(e1 - ref) - kLeanT + 127, 254), 0) : 0;
        if constexpr (V == kLeanP) {
          // bias per block: (C - 8e)/128, exact; a fully masked block has only
          // -inf scores, which give code 0 whatever the bias
          cb0 = v0 ? (kLeanC - 8.0f * e0) * (1.0f / 128.0f) : 0.0f;
          cb1 = v1 ? (kLeanC - 8.0f * e1) * (1.0f / 128.0f) : 0.0f;
        } else {
          // exponent x/8 - e + T = s*lam + (T - e); masked keys (-inf) give 0
          cb0 = v0 ? (float)kLeanT - e0 : 0.0f;
          cb1 = v1 ? (float)kLeanT - e1 : 0.0f;
        }
        // scale factor bytes: K-steps 0-1 (block 0) and 2-3 (block 1)
        sfa = (uint32_t)x0 | ((uint32_t)x0 << 8) | ((uint32_t)x1 << 16) | ((uint32_t)x1 << 24);
      } else {
        const float mt = fmaxf(block_max64(s, 0), block_max64(s, 64)) * lam;  // log2 units
        if (!have_ref) {
          ref = mt;
          have_ref = true;
        } else if (mt > ref) {
          alpha = ex2_approx(ref - mt);
          ref = mt;
          rescale = true;
        }
        cb0 = cb1 = -ref;
      }
      // The code step for words [W0, W1) of P (4 FP8 or 2 BF16 probabilities
      // per 32-bit word; words 0-15 hold the first 64-key block on FP8).
      auto codes = [&](auto w0c, auto w1c) {
        constexpr int W0 = decltype(w0c)::value, W1 = decltype(w1c)::value;
        if constexpr (V == kLeanP || V == kLeanPA3) {
#pragma unroll
          for (int w = W0; w < W1; ++w)
            pw[w] = leanp_codes4(__uint_as_float(s[4 * w]), __uint_as_float(s[4 * w + 1]),
                                 __uint_as_float(s[4 * w + 2]), __uint_as_float(s[4 * w + 3]),
                                 lamc, w < 16 ? cb0 : cb1, kc);
        } else if constexpr (V == kBlockExact) {
#pragma unroll
          for (int w = W0; w < W1; ++w) {
            const float g = w < 16 ? cb0 : cb1;
            float pv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = ex2_approx(fmaf(__uint_as_float(s[4 * w + i]), lam, g));
            pw[w] = f32x2_to_e4m3x2(pv[0], pv[1]) | (f32x2_to_e4m3x2(pv[2], pv[3]) << 16);
          }
        } else if constexpr (V == kExactFp8) {
#pragma unroll
          for (int w = W0; w < W1; ++w) {
            float pv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              pv[i] = ex2_approx(fmaf(__uint_as_float(s[4 * w + i]), lam, cb0));
            ls0 += pv[0] + pv[2];
            ls1 += pv[1] + pv[3];
            const uint32_t lo = f32x2_to_e4m3x2(pv[0], pv[1]);
            const uint32_t hi = f32x2_to_e4m3x2(pv[2], pv[3]);
            pw[w] = lo | (hi << 16);
          }
        } else {
#pragma unroll
          for (int w = W0; w < W1; ++w) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(s[2 * w]), lam, cb0));
            const float p1 = ex2_approx(fmaf(__uint_as_float(s[2 * w + 1]), lam, cb0));
            ls0 += p0;
            ls1 += p1;
            __nv_bfloat162 hv = __floats2bfloat162_rn(p0, p1);
            pw[w] = *reinterpret_cast<uint32_t*>(&hv);
          }
        }
      };
      // P_t(j-1) must have been consumed, and O_t must be final for j-1
      // before it is corrected for a raised reference.
      auto wait_o_and_rescale = [&]() -> bool {
        if (j > j0 && !warp_wait(&bars.o_done[t], (o_cnt - 1) & 1, ab, lim)) return false;
        if constexpr (V == kLeanPA3) {
          // frequent, non-power-of-two: 32-column passes with packed multiplies
          // (the second block's scores are still live here) and the row-sum column
          if (__any_sync(0xffffffffu, rescale)) {
            tc_fence_after();
            const uint64_t a2 = f32x2_pack(alpha, alpha);
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
              uint32_t o[32];
              tmem_ld32_wait(o_col + c, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const uint64_t y = mul_f32x2(f32x2_pack(__uint_as_float(o[2 * i]),
                                                        __uint_as_float(o[2 * i + 1])), a2);
                f32x2_unpack(y, o[2 * i], o[2 * i + 1]);
              }
              tmem_st32(o_col + c, o);
            }
            const float lv = __uint_as_float(tmem_ld1_wait(o_col + 128)) * alpha;
            tmem_st1(o_col + 128, __float_as_uint(lv));
          }
        } else if (__any_sync(0xffffffffu, rescale)) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t o[32];
            tmem_ld32_wait(o_col + c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(o_col + c, o);
          }
          if constexpr (C::kBlockScaled) {  // the row-sum column
            const float lv = __uint_as_float(tmem_ld1_wait(o_col + 128)) * alpha;
            tmem_st1(o_col + 128, __float_as_uint(lv));
          }
        }
        return true;
      };
      using W0 = std::integral_constant<int, 0>;
      using W16 = std::integral_constant<int, 16>;
      using W32 = std::integral_constant<int, 32>;
      if constexpr (C::kPHalves) {
        // first 64-key block: its codes and both blocks' scale factors, then
        // the P.V warp may issue K-steps 0-1 while the second block is coded
        codes(W0{}, W16{});
        if (stamp) FA8_TL(t, j, 3);
        if (!wait_o_and_rescale()) return;
        tmem_st16(p_col, *reinterpret_cast<uint32_t(*)[16]>(&pw[0]));
        tmem_st1(p_col + 32 + quad, sfa);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars.p_half[t]);
        codes(W16{}, W32{});
        tmem_st16(p_col + 16, *reinterpret_cast<uint32_t(*)[16]>(&pw[16]));
        if constexpr (!C::kBlockScaled) l = l * alpha + (ls0 + ls1);
      } else {
        codes(W0{}, std::integral_constant<int, C::kPCols>{});
        if constexpr (!C::kBlockScaled) l = l * alpha + (ls0 + ls1);
        if (stamp) FA8_TL(t, j, 3);
        if (!wait_o_and_rescale()) return;
        if constexpr (C::kFp8) {
          tmem_st32(p_col, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
          tmem_st1(p_col + 32 + quad, sfa);
        } else {
          tmem_st32(p_col, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
          tmem_st32(p_col + 32, *reinterpret_cast<uint32_t(*)[32]>(&pw[32]));
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars.p_full[t]);
      if (stamp) FA8_TL(t, j, 4);
      ++o_cnt;
    }
    if constexpr (C::kPrefetchItem) prefetch_item(round + 1);
    // epilogue: out = dv * O / l
    if (!warp_wait(&bars.o_done[t], (o_cnt - 1) & 1, ab, lim)) return;
    if (r == 0) FA8_TL(5, round, 4 * t + 1);
    tc_fence_after();
    const bool store = row < p.S;
    const size_t orow = ((size_t)b * p.S + (size_t)(row < p.S ? row : 0)) * p.Hq + h;
    // the reference in log2 units (the A3 path keeps it in raw-score units)
    const float ref2 = V == kLeanPA3 ? ref * lam : ref;
    // row sum l (relative to 2^ref): Lean-P paths, the scaled rounded weights
    // in O's row-sum column; exact paths, the unrounded p summed on the cores
    if constexpr (SPLIT) {
      // the piece is worked out again from the unit index here, so that the
      // key-tile loop carries one register for it instead of three
      const int ns = p.split_ns, sidx = w.u / ns, piece = w.u - sidx * ns;
      if (w.u < p.n_split_items * ns) {
        // One piece of a split item: O, l and ref (O and l relative to 2^ref)
        // go to the workspace and O_t is released; the piece that arrives
        // last adds the pieces up in piece order, rescaled to the largest
        // ref (Lean-P: integer binades, so the rescale is an exact power of
        // two; BF16: the running maxima, exp2 of their difference), so the
        // sum does not depend on which piece it is, and writes the output.
        // The others are done with this unit.
        float lt = l;  // exact paths: the unrounded row sum in registers
        if constexpr (C::kBlockScaled) lt = __uint_as_float(tmem_ld1_wait(o_col + 128));
        float* slots = reinterpret_cast<float*>(p.ws + split_cnt_bytes(p.n_split_items));
        auto slot = [&](int s_) {
          return slots + ((size_t)(sidx * ns + s_) * 2 + t) * kSplitSlotFloats;
        };
        float* mine = slot(piece);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {  // O in 32-column chunks
          uint32_t o[32];
          tmem_ld32_wait(o_col + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(reinterpret_cast<float4*>(mine) + (8 * c + i) * 128 + r,
                   make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                               __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3])));
        }
        tc_fence_before();
        mbar_arrive(&bars.o_free[t]);
        __stcg(mine + 128 * 128 + r, lt);
        __stcg(mine + 128 * 129 + r, ref2);
        __threadfence();
        // the tile's four warps: every row's partial is written and fenced
        // (an mbarrier, so that the wait is bounded like every other)
        auto group_sync = [&]() {
          mbar_arrive(&bars.split_sync[t]);
          return warp_wait(&bars.split_sync[t], (sync_cnt++) & 1, ab, lim);
        };
        if (!group_sync()) return;
        if (r == 0) bars.split_last[t] = split_arrive(p, sidx, ns, t, ab) ? 1 : 0;
        if (!group_sync()) return;
        if (!bars.split_last[t]) continue;
        __threadfence();
        // every piece from the workspace (this one's too), in piece order,
        // rescaled to the largest reference: the output straight from the
        // sums, 32 columns at a time (no 128-value array in registers)
        float R = -INFINITY;
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (s < ns) R = fmaxf(R, __ldcg(slot(s) + 128 * 129 + r));
        float sc[4];
        float L = 0.0f;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          sc[s] = 0.0f;
          if (s < ns) {
            const float d = __ldcg(slot(s) + 128 * 129 + r) - R;  // <= 0 (Lean-P: integers)
            if constexpr (C::kBlockScaled)
              sc[s] = d < -126.0f ? 0.0f : pow2i((int)d);
            else
              sc[s] = exp2f(d);
            L = fmaf(__ldcg(slot(s) + 128 * 128 + r), sc[s], L);
          }
        }
        const float inv = dvv / L;
        if (p.lse && store)
          p.lse[((size_t)b * p.Hq + h) * p.S + row] = (R + log2f(L)) * 0.6931471805599453f;
        // 32 output columns at a time: every piece's values are loaded
        // before any of the group's stores, so the loads of a group are in
        // flight together instead of waiting behind stores that might alias
        auto sum32 = [&](int g, float (&y)[32]) {  // columns 32g .. 32g+31
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = 0.0f;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            if (s < ns) {
              float4 x[8];
              const float4* src = reinterpret_cast<const float4*>(slot(s)) + (8 * g) * 128 + r;
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] = __ldcg(src + i * 128);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                y[4 * i] = fmaf(x[i].x, sc[s], y[4 * i]);
                y[4 * i + 1] = fmaf(x[i].y, sc[s], y[4 * i + 1]);
                y[4 * i + 2] = fmaf(x[i].z, sc[s], y[4 * i + 2]);
                y[4 * i + 3] = fmaf(x[i].w, sc[s], y[4 * i + 3]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] *= inv;
        };
        auto bf16x8 = [&](const float (&y)[32], int c) {  // y[8c .. 8c+7] as eight bf16
          uint32_t w4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 hv = __floats2bfloat162_rn(y[8 * c + 2 * k], y[8 * c + 2 * k + 1]);
            w4[k] = *reinterpret_cast<uint32_t*>(&hv);
          }
          return make_uint4(w4[0], w4[1], w4[2], w4[3]);
        };
        if (C::kEpiTma && !p.out_f32) {
          // as the whole-item epilogue below: this warp's slot, TMA stores
          uint8_t* oslot = smem + C::kSmemOut + (t * 4 + quad) * C::kOutSlotBytes;
          const int row0 = qb * 256 + t * 128 + (int)quad * 32;
          const uint32_t lane = lane_id();
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float y0[32], y1[32];
            sum32(2 * half, y0);
            sum32(2 * half + 1, y1);
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              *reinterpret_cast<uint4*>(oslot + lane * 128 + ((c ^ (lane & 7)) * 16)) = bf16x8(y0, c);
              *reinterpret_cast<uint4*>(oslot + lane * 128 + (((c + 4) ^ (lane & 7)) * 16)) =
                  bf16x8(y1, c);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < p.S) {
              tma_store_4d(&maps.o64, oslot, 64 * half, h, row0, b);
              bulk_commit();
            }
          }
        } else if (store) {
#pragma unroll 1
          for (int g = 0; g < 4; ++g) {
            float y[32];
            sum32(g, y);
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kDV) + 8 * g;
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDV) + 4 * g;
#pragma unroll
              for (int c = 0; c < 4; ++c) dst[c] = bf16x8(y, c);
            }
          }
        }
        continue;
      }
    }
    if constexpr (C::kEarlyOFree) {
      // O_t (and its row-sum column) in registers with one wait, then O_t is
      // released before the stores, so the next item's first P.V product
      // does not wait for them
      uint32_t o[128];
      uint32_t lsum;
      tmem_ld128_1_wait(o_col, o_col + (C::kBlockScaled ? 128 : 0), o, lsum);
      tc_fence_before();
      mbar_arrive(&bars.o_free[t]);
      if (r == 0) FA8_TL(5, round, 4 * t + 2);
      if constexpr (C::kBlockScaled) l = __uint_as_float(lsum);
      const float inv = dvv / l;
      if (p.lse && store)
        p.lse[((size_t)b * p.Hq + h) * p.S + row] = (ref2 + log2f(l)) * 0.6931471805599453f;
      if (C::kEpiTma && !p.out_f32) {
        // bf16 rows through this warp's shared-memory slot and TMA stores (the
        // tensor map clips rows past S): the warp does not wait for global
        // memory, only for the slot's previous contents to have been read.
        // The normalisation runs on packed pairs (measured 0.2-2.5% faster
        // than scalar multiplies, most at short sequences).
        uint8_t* slot = smem + C::kSmemOut + (t * 4 + quad) * C::kOutSlotBytes;
        const int row0 = qb * 256 + t * 128 + (int)quad * 32;
        const uint32_t lane = lane_id();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16-byte chunk c: columns 64*half + 8c .. +7
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int col = 64 * half + 8 * c + 2 * k;
              uint32_t x0, x1;
              f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(o[col]), __uint_as_float(o[col + 1])),
                                     f32x2_pack(inv, inv)), x0, x1);
              __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(x0), __uint_as_float(x1));
              w[k] = *reinterpret_cast<uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(slot + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.S) {  // a box wholly past S stores nothing
            tma_store_4d(&maps.o64, slot, 64 * half, h, row0, b);
            bulk_commit();
          }
        }
      } else if (store) {
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kDV);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv,
                                 __uint_as_float(o[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDV);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(o[8 * i + 2 * k]) * inv,
                                                        __uint_as_float(o[8 * i + 2 * k + 1]) * inv);
              w[k] = *reinterpret_cast<uint32_t*>(&hv);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (r == 0) FA8_TL(5, round, 4 * t + 3);
    } else {
      if constexpr (C::kBlockScaled) l = __uint_as_float(tmem_ld1_wait(o_col + 128));
      const float inv = dvv / l;
      if (p.lse && store)
        p.lse[((size_t)b * p.Hq + h) * p.S + row] = (ref2 + log2f(l)) * 0.6931471805599453f;
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        uint32_t o[32];
        tmem_ld32_wait(o_col + c, o);
        if (store) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow * kDV + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                   __uint_as_float(o[4 * i + 2]) * inv,
                                   __uint_as_float(o[4 * i + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow * kDV + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                __nv_bfloat162 hv = __floats2bfloat162_rn(__uint_as_float(o[8 * i + 2 * k]) * inv,
                                                          __uint_as_float(o[8 * i + 2 * k + 1]) * inv);
                w[k] = *reinterpret_cast<uint32_t*>(&hv);
              }
              dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars.o_free[t]);
    }
  }
}

// --------------------------------------------------------------------------
// The kernel.
// --------------------------------------------------------------------------
template <int V, int DQK, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ Maps maps, const KParams p) {
  using C = Cfg<V, DQK>;
  // the split schedule: Lean-P and block-exact, whose codes depend on each
  // 64-key block alone (a split changes only the order of the fp32 sums),
  // and BF16, whose probabilities are rounded relative to each piece's own
  // running maximum (within the rounding of bf16)
  static_assert(!SPLIT || V == kLeanP || V == kBlockExact || V == kBf16,
                "split units: block-local codes or bf16 probabilities");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ Barriers bars;
  const uint32_t warp = warp_id();
  if (threadIdx.x == 0) {
    bars.abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.s_drained[t], 128);
      mbar_init(&bars.p_full[t], 128);
      mbar_init(&bars.p_half[t], 128);
      mbar_init(&bars.o_done[t], 1);
      for (int i = 0; i < 4; ++i) mbar_init(&bars.qk_go[t][i], 1);
      mbar_init(&bars.o_free[t], 128);
      mbar_init(&bars.drain[t], 1);
      mbar_init(&bars.split_sync[t], 128);
    }
    fence_mbar_init();
  }
  if constexpr (C::kOnesBytes > 0) {
    // the ones atom of the P.V B operand: e4m3 1.0 everywhere
    uint4* ones = reinterpret_cast<uint4*>(smem + C::kSmemOnes);
    for (int i = threadIdx.x; i < C::kOnesBytes / 16; i += kThreads)
      ones[i] = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
    fence_proxy_async_smem();
  }
  if (warp == kPvWarp) {
    tmem_alloc(&bars.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  if constexpr (C::kFp8) {
    // B-operand scale factors of every P.V product: 1.0 (never overwritten)
    if (warp < 4) {
      tmem_st4(tmem + ((warp * 32) << 16) + C::kColSfb, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu,
               0x7F7F7F7Fu);
      tmem_st1(tmem + ((warp * 32) << 16) + C::kColSfb + 4, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (warp < 8) {
    softmax_loop<V, DQK, SPLIT>(p, maps, smem, bars, tmem, warp / 4);
    // bulk stores of the output must be complete before the CTA exits
    if (C::kEpiTma && lane_id() == 0) bulk_wait_all();
    __syncwarp();
  } else if (warp == kProducerWarp) {
    producer_loop<V, DQK, SPLIT>(p, maps, smem, bars);
  } else if (warp == kQkWarp || warp == kPvWarp) {
    const int role = warp == kQkWarp ? 0 : 1;
    if (role == 0)
      qk_loop<V, DQK, SPLIT>(p, smem_u32(smem), bars, tmem);
    else
      pv_loop<V, DQK, SPLIT>(p, smem_u32(smem), bars, tmem);
    if (lane_id() == 0) {
      // every MMA this thread issued must be complete before TMEM is released;
      // a drain that runs out of time is reported like any other expired wait
      volatile int gave_up = 0;
      tc_commit(&bars.drain[role]);
      if (!mbar_wait(&bars.drain[role], 0, &gave_up, 50000000ull))
        *reinterpret_cast<volatile int*>(&bars.abort_flag) = 1;
    }
    __syncwarp();
  }

  // Teardown: the producer has waited for its last copies (on every exit) and
  // each MMA warp for its MMAs; an expired wait anywhere sets the status word.
  tc_fence_before();
  __syncthreads();
  if (bars.abort_flag && threadIdx.x == 0 && p.status) atomicExch(p.status, 5);
  if (warp == kPvWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa8
