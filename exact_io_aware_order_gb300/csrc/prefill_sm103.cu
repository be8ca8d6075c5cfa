// Causal (or full) prefill attention forward, sm_103a: TMA + tcgen05 + TMEM.
//
// Page "FlashAttention for inference: tiled prefill and split-KV decoding",
// section "Prefill: tiles, loop order and the tensor cores": the outer,
// parallel loop runs over (sequence, head, query tile); each block loads its
// query tile once, streams key/value tiles up to the causal limit through
// on-chip memory, computes S = Q_i K_j^T * scale on the tensor cores (masking
// only the diagonal tile), updates the running max m and sum l with the
// correction c = exp(m_old - m_new) (section "The online softmax, with every
// symbol defined"), accumulates acc = c*acc + P V_j on the tensor cores, and
// finally writes O_i = acc / l and the row log-sum-exp m + log l.  Tiles
// strictly above the diagonal are never visited.
//
// GB300 design (the pages' A100/H100 kernels are prior art only):
//   * persistent CTAs, one per SM, each walking its share of a work list of
//     128-row query tiles (longest causal rows first, snake order across
//     CTAs); every role counts tiles over all items, so the pipeline does not
//     drain between items;
//   * key/value tiles of 128 keys (64 at head_dim 256), streamed by TMA
//     (128-byte swizzle, 3-D tensor maps so rows past the end read as zero)
//     into a K ring and a V ring in shared memory; Q tiles double-buffered;
//   * TMEM (512 columns): S buffers and O accumulators (see s_bufs / o_bufs):
//     three S buffers and one O in bf16 at head_dim 128, so the tensor core
//     computes S(j+1), S(j+2) while the softmax works on S(j); two O (items
//     alternating) at head_dim 64 and in FP8.
//     P(j) is written as bf16 over the first half of S(j)'s buffer and feeds
//     O += P V straight from TMEM (A operand in tensor memory), V from shared
//     memory (MN-major);
//   * two threads issue tcgen05.mma: warp 5 the S products (S(j) as soon as
//     K_j is in and the P V product that last read its buffer has finished),
//     warp 6 the P V products (as soon as P(j) and V_j are ready).  Every
//     wait or commit stalls its issuing thread for longer than one
//     128x128x16 MMA runs, so one thread alone leaves the tensor core idle
//     between groups; with two, one thread's synchronisation overlaps the
//     other's MMAs.  Warp 4 is the TMA producer;
//   * warps 0-3 run the softmax, one query row per thread (TMEM lane = row),
//     so row max and row sum need no shuffles and no cross-warp exchange;
//   * warps 7-10 are the epilogue: O / l read from TMEM once the item's last
//     product is done (O is released at once for the next item), written
//     through swizzled shared-memory boxes by TMA stores, and the LSE;
//   * base-2 exponentials with scale*log2(e) folded in; O is rescaled only
//     when a row max grows by more than 2^8 (the same stale max is used for
//     l and O, so the result is exact), and only after the previous P V
//     product has completed; the LSE is converted back to natural log;
//   * flavours compiled separately, so the plain kernel carries none of the
//     others' code: sliding window, window and/or soft-capping, ALiBi (with
//     an optional window), FP8 (e4m3 operands, kind::f8f6f4, per-block
//     scales), each padded or packed (variable-length sequences), and each
//     with an fp32 or a bf16 O;
//   * every wait is bounded; on a timeout all roles leave their loops, the
//     CTA waits for in-flight copies and MMAs, frees TMEM and exits.
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;                 // rows per query tile
// Keys per key/value tile: 128, or 64 for head_dim 256 (three S buffers of
// 64 columns and O's 256 columns then fit the 512 TMEM columns).
template <int D>
constexpr int key_tile() { return D == 256 ? 64 : 128; }

// TMEM buffers: SB S buffers (kBN columns each; P aliases S) and OB O
// accumulators (D columns each), within 512 columns.  With two O buffers an
// item's first P V product need not wait for the epilogue to read the last
// item's O; two S buffers make S(j + 2) wait for P V(j).  head_dim 64: three
// S and two O (384 + 128).  128: three S and one O (384 + 128) in bf16, where
// the softmax leaves the S-after-P V chain too little slack (measured 15%
// slower with two and two); two S and two O (256 + 256) in FP8, whose halved
// products leave enough (measured 1.3% faster).  256: three S of 64 keys and
// one O (192 + 256).
template <int D, bool FP8>
__host__ __device__ constexpr int s_bufs() {
  return (D == 128 && FP8) ? 2 : 3;
}
template <int D, bool FP8>
__host__ __device__ constexpr int o_bufs() {
  return (D == 256 || (D == 128 && !FP8)) ? 1 : 2;
}
constexpr int kThreads = 352;            // 11 warps
constexpr int kSoftmaxThreads = 128;     // warps 0-3: one query row per thread
constexpr int kProducerWarp = 4;
constexpr int kSWarp = 5;                // issues S = Q K^T
constexpr int kPVWarp = 6;               // issues O += P V
constexpr int kEpiWarp0 = 7;             // warps 7-10: O / LSE epilogue
constexpr int kEpiThreads = 128;
constexpr int kSBuf = 3;                 // most S buffers in TMEM (barrier layout)
constexpr int kOBufMax = 2;              // most O buffers in TMEM (barrier layout)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when max grows > 2^8

// ESZ: bytes per element of Q, K and V (2: bf16; 1: e4m3).  XB: the ALiBi
// bias's extra k-step operands (two constant 4 KB key chunks, a 256-byte
// query atom per Q slot).
template <int D, bool VARLEN, int ESZ = 2, bool XB = false>
struct PrefillSmem {
  static constexpr int kBNt = key_tile<D>();
  static constexpr int kQTileBytes = 128 * D * ESZ;    // one Q tile (128 rows)
  static constexpr int kTileBytes = kBNt * D * ESZ;    // one K or V tile
  static constexpr int kQChunkBytes = 128 * 128;       // 128 rows x 128 B (one swizzle span)
  static constexpr int kChunkBytes = kBNt * 128;       // K / V: kBNt rows x 128 B
  static constexpr int kChunks = D * ESZ / 128;        // swizzle spans per row
  static constexpr int kQSlots = D == 256 ? 1 : 2;     // a 64 KB Q tile leaves room for one
  static constexpr int kKSlots = kTileBytes == 32768 ? 2 : 4;
  static constexpr int kVSlots = kTileBytes == 32768 ? 2 : 6;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQSlots * kQTileBytes;
  static constexpr int kV = kK + kKSlots * kTileBytes;
  static constexpr int kStage = kV + kVSlots * kTileBytes;     // O staging: 4 warps x 32 rows x 128 B
  // ALiBi: K'+ and K'- (128 rows x 32 B each), then Q' per Q slot (8 rows x
  // 32 B: all 128 rows of Q' are equal, so its 8-row groups share one atom).
  static constexpr int kKxPos = kStage + 4 * 4096;
  static constexpr int kKxNeg = kKxPos + 4096;
  static constexpr int kQx = kKxNeg + 4096;
  static constexpr int kQxBytes = 256;
  static constexpr int kBar = kKxPos + (XB ? 2 * 4096 + kQSlots * kQxBytes : 0);
  static_assert(!XB || (kKxNeg == kKxPos + 4096 && kQx + kQSlots * kQxBytes == kBar),
                "ALiBi operand layout");
  // barriers: q_full/q_empty, k_full/k_empty, v_full/v_empty (one pair per
  // slot), s_full/p_full/pv_done [3], o_full, o_empty, stats_full/stats_empty [2],
  // drain_s, drain_pv
  static constexpr int kNumBars =
      2 * kQSlots + 2 * kKSlots + 2 * kVSlots + 3 * kSBuf + 2 * kOBufMax + 4 + 2;
  static constexpr int kStats = kBar + kNumBars * 8;           // float2 (m, l) [2][128]
  static constexpr int kMisc = kStats + 2 * 128 * 8;           // tmem base, abort flag
  // Packed variable-length mode: per sequence its first row, its length and
  // the running count of work items before it (one more entry: the total).
  static constexpr int kSeqStart = kMisc + 16;
  static constexpr int kSeqLen = kSeqStart + (VARLEN ? kMaxVarlenSeqs * 4 : 0);
  static constexpr int kItemPrefix = kSeqLen + (VARLEN ? kMaxVarlenSeqs * 4 : 0);
  static constexpr int kUsed = kItemPrefix + (VARLEN ? (kMaxVarlenSeqs + 1) * 4 : 0);
  static constexpr int kAlloc = kUsed + 1024;                  // + alignment slack
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct PrefillParams {
  void* o;          // fp32, or bf16 in the OBF16 kernels
  float* lse;
  int batch, n_q_heads, n_kv_heads, seqlen;
  float sl2;  // scale * log2(e); with soft-capping, softcap * log2(e)
  int causal;
  int window_left;  // sliding window: row i sees keys j >= i - window_left (-1: none)
  float cap_in2;    // soft-capping: 2 log2(e) scale / softcap (the tanh argument's factor)
  const float* alibi_slopes;  // ALiBi: per query head slope (natural-log units)
  int n_q_tiles;    // ceil(seqlen / 128)
  int total_tiles;  // n_q_tiles * batch * n_q_heads (padded mode)
  int group_planes; // plain padded mode: query planes per kv-head group of the work list
  const int32_t* cu_seqlens;  // packed mode: (num_seqs + 1) row offsets
  int num_seqs;
  int seq_base;     // packed mode: cu_seqlens[0]'s index in the caller's list
  // FP8: dequantisation scales of the e4m3 inputs, per 128-row block of Q and
  // K ((plane, n_q_tiles)) and per head of V ((plane,)).
  const float* q_scales;
  const float* k_scales;
  const float* v_scales;
  // FP8: O's columns (head_dim 64 or 128).  At 64 the copies of Q, K and V^T
  // fill the tiles' second half with zeros, which add nothing to S and give
  // zero columns 64..127 of O; only the first 64 are stored.
  int d_out;
  uint32_t* err_word;
  uint64_t timeout_ns;
};

// One query tile of one (sequence, head).
struct Tile {
  int row0;  // tensor-map row of the tile's first query
  int qrel;  // index of that query within its sequence
  int kv0;   // tensor-map row of the sequence's first key
  int len;   // sequence length (keys and queries)
  int zq;    // Q / O tensor-map plane (sequence * n_q_heads + head)
  int zk;    // K / V tensor-map plane
  int j0;    // first key tile visited (> 0 only with a sliding window)
  int n;     // key tiles visited (>= 1)
  int tile0; // FP8 scales: the sequence's first 128-row tile in the scale arrays
};

// Shared-memory tables of the packed variable-length mode.
struct SeqTables {
  const int* start;   // first row of each sequence
  const int* len;     // length of each sequence
  const int* prefix;  // work items before each sequence; prefix[num_seqs] = all items
};

// Work list, longest causal rows first.  Padded batch: item w is query tile
// n_q_tiles - 1 - w / (batch * n_q_heads) of (sequence, head) w % (batch * n_q_heads),
// so consecutive items share kv heads while their K/V tiles are hot in L2.
// Packed sequences: the items of sequence s are prefix[s] .. prefix[s+1]-1,
// again longest tile first and heads fastest, taken in the same snake order,
// so the CTAs work on one or two sequences at a time and their K/V stay in
// L2.  (A globally longest-first order balances better but spreads the work
// over every sequence at once; claiming items dynamically balances too but
// costs more per tile; both measured slower.)
// Kernel flavours: the plain kernel, one with a sliding window, one with a
// window and / or soft-capping, one with ALiBi and an optional window (the
// window and the cap are set at run time).
enum Variant : int { kPlain = 0, kWindow = 1, kWindowCap = 2, kWindowAlibi = 3, kFp8 = 4 };

template <bool VARLEN, int VARIANT, int kBN>
__device__ __forceinline__ Tile tile_of(int w, const PrefillParams& p, const SeqTables& st) {
  Tile t;
  if constexpr (!VARLEN) {
    int qt, bh;
    if constexpr (VARIANT == kPlain) {
      // The list runs over groups of group_planes consecutive query planes
      // (whole kv heads), each group's items longest first with heads
      // fastest, and every other group in the opposite direction so that
      // lengths do not jump at group boundaries (the snake order below then
      // still balances).  With one group (the whole batch) this is the plain
      // longest-first order; several groups keep only a few kv heads' K/V in
      // use at a time, so that they stay in L2 when all of them would not
      // fit.  (Only this flavour: the others run close to their register
      // limit, and the extra index arithmetic measured slower there.)
      const int P = p.batch * p.n_q_heads;
      const int grp = w / (p.n_q_tiles * p.group_planes);
      const int local = w - grp * p.n_q_tiles * p.group_planes;
      const int gh = min(p.group_planes, P - grp * p.group_planes);
      const int rank = local / gh;
      qt = (grp & 1) ? rank : p.n_q_tiles - 1 - rank;
      bh = grp * p.group_planes + local % gh;
    } else {
      const int BH = p.batch * p.n_q_heads;
      qt = p.n_q_tiles - 1 - w / BH;
      bh = w % BH;
    }
    const int bidx = bh / p.n_q_heads, h = bh % p.n_q_heads;
    const int kvh = h / (p.n_q_heads / p.n_kv_heads);
    t.row0 = t.qrel = qt * kBM;
    t.kv0 = 0;
    t.len = p.seqlen;
    t.zq = bidx * p.n_q_heads + h;
    t.zk = bidx * p.n_kv_heads + kvh;
    t.tile0 = 0;
    t.n = p.causal ? (qt + 1) * kBM / kBN : (p.seqlen + kBN - 1) / kBN;
  } else {
    // The sequence: the last one whose first item is at or before w (a
    // sequence without items shares its prefix with the next one).
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (st.prefix[mid] <= w) lo = mid; else hi = mid - 1;
    }
    const int local = w - st.prefix[lo];
    const int h = local % p.n_q_heads;
    const int tiles = (st.len[lo] + kBM - 1) / kBM;
    const int qt = tiles - 1 - local / p.n_q_heads;
    t.qrel = qt * kBM;
    t.row0 = st.start[lo] + t.qrel;
    t.kv0 = st.start[lo];
    t.len = st.len[lo];
    t.zq = h;
    t.zk = h / (p.n_q_heads / p.n_kv_heads);
    t.tile0 = st.prefix[lo] / p.n_q_heads;  // items per sequence = its tiles x heads
    t.n = p.causal ? (qt + 1) * kBM / kBN : (t.len + kBN - 1) / kBN;
  }
  // A sliding window skips the key tiles left of every row's window: the
  // tile's first row sees keys from qrel - window_left on.
  t.j0 = 0;
  if constexpr (VARIANT != kPlain) {
    if (p.window_left >= 0 && t.qrel > p.window_left) t.j0 = (t.qrel - p.window_left) / kBN;
    t.n -= t.j0;
  }
  return t;
}

// The key tile an item visits j-th: in order, or, for causal ALiBi, from the
// diagonal backwards.  The ALiBi bias grows toward the diagonal, so in order
// the running max would grow tile after tile and O would be rescaled nearly
// every tile; backwards, the first tile holds the row's largest scores.  The
// online softmax is exact in any order.
template <int VARIANT>
__device__ __forceinline__ int key_tile_at(const Tile& t, int j, int causal) {
  return (VARIANT == kWindowAlibi && causal) ? t.j0 + t.n - 1 - j : t.j0 + j;
}

// The r-th item of this CTA, or -1: rounds of gridDim.x items, taken in
// alternating (snake) order so that, over two rounds, every CTA gets about
// the same number of key tiles.
__device__ __forceinline__ int item_of(int r, int total) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int w = r * G + ((r & 1) ? (G - 1 - c) : c);
  return w < total ? w : -1;
}

// VARIANT selects the flavour (see Variant): the plain kernel has neither a
// window nor soft-capping in its code, the window kernel no soft-capping.
// OBF16: O is written as bf16 (acc / l in fp32, rounded once); a template
// parameter, so that the fp32 kernels carry none of that code.
template <int D, bool VARLEN, int VARIANT, bool OBF16>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const PrefillParams p) {
  constexpr bool FP8 = VARIANT == kFp8;
  constexpr int kBN = key_tile<D>();
  constexpr int SB = s_bufs<D, FP8>(), OB = o_bufs<D, FP8>();
  static_assert(SB <= kSBuf && OB <= kOBufMax && SB * kBN + OB * D <= (int)kTmemCols,
                "TMEM budget");
  // ALiBi at head_dim <= 128: the tensor core adds the bias's per-key part.
  constexpr bool XB = VARIANT == kWindowAlibi && D <= 128;
  // Edge tiles: masked per 32-column chunk, with a warp-wide test first (the
  // warp's rows are consecutive, so its smallest last-allowed column is its
  // first row's and its largest first-allowed column its last row's; a chunk
  // inside both for every row needs no per-score test), or per score.  Which
  // form schedules better depends on the flavour: measured, the chunked form
  // is faster in the plain and soft-capping flavours, slower in the others.
  constexpr bool kChunkMask = (VARIANT == kPlain && !VARLEN) || VARIANT == kWindowCap;
  using L = PrefillSmem<D, VARLEN, FP8 ? 1 : 2, XB>;
  constexpr int RQ = L::kQSlots, RK = L::kKSlots, RV = L::kVSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.seqlen;

  // Barrier layout.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int kQFull = 0, kQEmpty = kQFull + RQ, kKFull = kQEmpty + RQ, kKEmpty = kKFull + RK,
            kVFull = kKEmpty + RK, kVEmpty = kVFull + RV, kSFull = kVEmpty + RV,
            kPFull = kSFull + kSBuf, kPVDone = kPFull + kSBuf, kOFull = kPVDone + kSBuf,
            kOEmpty = kOFull + kOBufMax, kStFull = kOEmpty + kOBufMax, kStEmpty = kStFull + 2,
            kDrainS = kStEmpty + 2, kDrainPV = kDrainS + 1;
  float2* stats = reinterpret_cast<float2*>(smem + L::kStats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc + 4);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < RQ; ++i) {
      mbar_init(bar(kQFull + i), 1);
      mbar_init(bar(kQEmpty + i), 1);
    }
    for (int i = 0; i < RK; ++i) {
      mbar_init(bar(kKFull + i), 1);
      mbar_init(bar(kKEmpty + i), 1);
    }
    for (int i = 0; i < RV; ++i) {
      mbar_init(bar(kVFull + i), 1);
      mbar_init(bar(kVEmpty + i), 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kPFull + i), kSoftmaxThreads);
      mbar_init(bar(kPVDone + i), 1);
    }
    for (int i = 0; i < OB; ++i) {
      mbar_init(bar(kOFull + i), 1);
      mbar_init(bar(kOEmpty + i), kEpiThreads);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kStFull + i), kSoftmaxThreads);
      mbar_init(bar(kStEmpty + i), kEpiThreads);
    }
    mbar_init(bar(kDrainS), 1);
    mbar_init(bar(kDrainPV), 1);
    fence_mbar_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_o);
  }
  int* seq_start = reinterpret_cast<int*>(smem + L::kSeqStart);
  int* seq_len = reinterpret_cast<int*>(smem + L::kSeqLen);
  int* item_prefix = reinterpret_cast<int*>(smem + L::kItemPrefix);
  if constexpr (VARLEN) {
    // Packed sequences: one warp reads cu_seqlens, clamps each sequence to
    // [previous end, total] (flagging any that had to be), and scans the
    // per-sequence item counts (n_q_heads x query tiles).
    if (warp == kEpiWarp0) {
      int carry = 0, prev_end = 0;
      bool bad = false, misaligned = false;
      for (int base = 0; base < p.num_seqs; base += 32) {
        const int s = base + lane;
        int a = 0, e = 0;
        if (s < p.num_seqs) {
          a = p.cu_seqlens[s];
          e = p.cu_seqlens[s + 1];
        }
        const int a_prev = __shfl_up_sync(0xffffffffu, e, 1);
        const int lower = lane == 0 ? prev_end : a_prev;  // the previous sequence's end
        int a_c = min(max(a, 0), N), e_c = min(max(e, a_c), N);
        // (only the list's first entry must be 0: a later slice starts where
        // the previous launch's last sequence ended)
        if (s < p.num_seqs &&
            (a != a_c || e != e_c || a < lower || (s == 0 && p.seq_base == 0 && a != 0)))
          bad = true;
        // FP8: V^T's copies take tokens along the innermost coordinate, which
        // a TMA copy of bytes needs at a multiple of 16: every non-empty
        // sequence must start there (else the launch does nothing, flagged).
        if (FP8 && s < p.num_seqs && e_c > a_c && (a_c & 15) != 0) misaligned = true;
        if (s >= p.num_seqs) a_c = e_c = 0;
        const int items = ((e_c - a_c + kBM - 1) / kBM) * p.n_q_heads;
        int incl = items;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        if (s < p.num_seqs) {
          seq_start[s] = a_c;
          seq_len[s] = e_c - a_c;
          item_prefix[s + 1] = carry + incl;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
        prev_end = __shfl_sync(0xffffffffu, e, 31);
      }
      if (lane == 0) item_prefix[0] = 0;
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err_word, kErrSeqLens);
      if (__any_sync(0xffffffffu, misaligned)) {
        for (int s = lane; s <= p.num_seqs; s += 32) item_prefix[s] = 0;  // no work, no copies
        if (lane == 0) atomicOr(p.err_word, kErrSeqLens);
      }
    }
  }
  if constexpr (XB) {
    // ALiBi's key chunks K'+ and K'-: row r (a key's offset in its tile) is
    // 32 bytes, two equal 16-byte halves of bf16 (+-r, +-r, +-r, 0, 0, 0, 0, 0),
    // so that any 32-byte swizzle of the halves reads the same values.
    for (int i = threadIdx.x; i < 2 * 256; i += kThreads) {
      const int which = i >> 8, u = i & 255, r = u >> 1;
      const float v = which ? -static_cast<float>(r) : static_cast<float>(r);
      st_shared_v4(smem_u32(smem + (which ? L::kKxNeg : L::kKxPos) + u * 16),
                   make_float4(__uint_as_float(pack_bf16x2(v, v)), __uint_as_float(pack_bf16x2(v, 0.f)),
                               0.f, 0.f));
    }
    fence_proxy_async_smem();  // read by the MMAs (async proxy)
  }
  const SeqTables seqt{seq_start, seq_len, item_prefix};
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: SB S buffers of kBN columns, then OB O buffers of D columns
  // (item r accumulates into O buffer r % OB, so with two the next item's
  // products need not wait for the epilogue to read the last item's O).
  const uint32_t tO = tmem + (uint32_t)(SB * kBN);
  auto o_buf = [&](int r) { return tO + (uint32_t)((r % OB) * D); };
  const WaitCtl ctl{abort_flag, p.err_word, p.timeout_ns};
  const int total = VARLEN ? item_prefix[p.num_seqs] : p.total_tiles;

  // Every role walks the same sequence: the CTA's items r = 0, 1, ... and,
  // within item r, key tiles j = 0 .. n-1.  Ring slots and barrier phases
  // follow the running count over all items (g for key tiles), so the
  // pipeline does not drain between items.
  // bf16: Q, K K-major, V MN-major.  e4m3: all K-major (V arrives transposed).
  const uint32_t id_s = FP8 ? idesc_e4m3_f32(kBM, kBN) : idesc_bf16_f32(kBM, kBN, false, false);
  const uint32_t id_pv = FP8 ? idesc_e4m3_f32(kBM, D) : idesc_bf16_f32(kBM, D, false, true);
  const uint32_t dhi = sw128_desc_hi(1024);

  if (warp == kProducerWarp) {
    // ============================ TMA producer ============================
    // Two cursors over the flattened (item, key tile) sequence: K runs two
    // key tiles ahead of V, and Q of an item is loaded just before its first
    // K, so the tiles arrive in the order the issuing threads consume them,
    // across item boundaries too.  A slot is reused once the MMAs that read
    // its previous tile have completed.
    if (lane == 0) {
      struct Cursor {
        int r, j, w;
        Tile t;
      };
      auto start = [&](Cursor& c) {
        c.r = 0;
        c.j = 0;
        c.w = item_of(0, total);
        if (c.w >= 0) c.t = tile_of<VARLEN, VARIANT, kBN>(c.w, p, seqt);
      };
      auto advance = [&](Cursor& c) {
        if (++c.j == c.t.n) {
          c.j = 0;
          c.w = item_of(++c.r, total);
          if (c.w >= 0) c.t = tile_of<VARLEN, VARIANT, kBN>(c.w, p, seqt);
        }
      };
      int nq = 0, nk = 0, nv = 0;  // tiles issued
      // `row`: first row of the tile in the tensor; a transposed tile (FP8
      // V, (plane, d, rows)) takes its rows along the innermost dimension.
      // L2 policy: Q is read once (evict first); K and V tiles are read again
      // by the other query tiles of their kv head (evict last).
      const uint64_t pol_once = l2_policy_evict_first(), pol_keep = l2_policy_evict_last();
      auto load_tile = [&](const CUtensorMap* map, int base, int full, int empty, int R, int cnt,
                           int row, int z, bool transposed) -> bool {
        const int slot = cnt % R;
        const bool is_q = base == L::kQ;
        const uint64_t pol = is_q ? pol_once : pol_keep;
        const int tile_bytes = is_q ? L::kQTileBytes : L::kTileBytes;
        const int chunk_bytes = is_q ? L::kQChunkBytes : L::kChunkBytes;
        if (cnt >= R && !mbar_wait(bar(empty + slot), ((cnt / R) - 1) & 1, ctl)) return false;
        if constexpr (XB) {
          if (is_q) {
            // ALiBi's query atom Q' for this slot: every row (h, m, l, 0, ...) / 2
            // in both 16-byte halves, where h + m + l (three bf16 terms) is
            // slope log2(e) / (scale log2(e)), so that Q' K'+- scaled by
            // scale log2(e) is +- slope (j - kv0) log2(e).
            const float tgt = p.alibi_slopes[z % p.n_q_heads] * kLog2e / p.sl2;
            const float h = bf16_round(tgt), mid = bf16_round(tgt - h), lo = bf16_round(tgt - h - mid);
            const float4 u = make_float4(__uint_as_float(pack_bf16x2(0.5f * h, 0.5f * mid)),
                                         __uint_as_float(pack_bf16x2(0.5f * lo, 0.f)), 0.f, 0.f);
            const uint32_t qx = smem_u32(smem + L::kQx + slot * L::kQxBytes);
            for (int i = 0; i < L::kQxBytes / 16; ++i) st_shared_v4(qx + i * 16, u);
            fence_proxy_async_smem();  // visible to the MMAs before the slot is announced
          }
        }
        mbar_arrive_expect_tx(bar(full + slot), (uint32_t)tile_bytes);
        for (int c = 0; c < L::kChunks; ++c) {
          const uint32_t dst = smem_u32(smem + base + slot * tile_bytes + c * chunk_bytes);
          if (transposed)
            tma_load_3d_hint(dst, map, bar(full + slot), row, c * 128, z, pol);
          else
            tma_load_3d_hint(dst, map, bar(full + slot), c * (128 / (FP8 ? 1 : 2)), row, z, pol);
        }
        return true;
      };
      Cursor kc, vc;
      start(kc);
      start(vc);
      auto load_k = [&]() -> bool {
        if (kc.w < 0) return true;
        if (kc.j == 0) {
          if (!load_tile(&tm_q, L::kQ, kQFull, kQEmpty, RQ, nq, kc.t.row0, kc.t.zq, false))
            return false;
          ++nq;
        }
        if (!load_tile(&tm_k, L::kK, kKFull, kKEmpty, RK, nk,
                       kc.t.kv0 + key_tile_at<VARIANT>(kc.t, kc.j, p.causal) * kBN,
                       kc.t.zk, false))
          return false;
        ++nk;
        advance(kc);
        return true;
      };
      bool ok = load_k() && load_k();
      while (ok && vc.w >= 0) {
        ok = load_tile(&tm_v, L::kV, kVFull, kVEmpty, RV, nv,
                       vc.t.kv0 + key_tile_at<VARIANT>(vc.t, vc.j, p.causal) * kBN,
                       vc.t.zk, FP8);
        if (!ok) break;
        ++nv;
        advance(vc);
        ok = load_k();
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's memory is released.
        volatile uint32_t no_abort = 0u;
        WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
        for (int i = max(0, nq - RQ); i < nq; ++i) mbar_wait(bar(kQFull + i % RQ), (i / RQ) & 1, drain);
        for (int i = max(0, nk - RK); i < nk; ++i) mbar_wait(bar(kKFull + i % RK), (i / RK) & 1, drain);
        for (int i = max(0, nv - RV); i < nv; ++i) mbar_wait(bar(kVFull + i % RV), (i / RV) & 1, drain);
      }
    }
  } else if (warp == kSWarp) {
    // ============================ S = Q K^T issuer ============================
    if (lane == 0) {
      const uint32_t k_lo0 = sw128_desc_lo(smem_u32(smem + L::kK), 16);
      bool ok = true;
      int g = 0;
      for (int r = 0; ok; ++r) {
        const int w = item_of(r, total);
        if (w < 0) break;
        const Tile t = tile_of<VARLEN, VARIANT, kBN>(w, p, seqt);
        const int qs = r % RQ;
        if (!mbar_wait(bar(kQFull + qs), (r / RQ) & 1, ctl)) { ok = false; break; }
        const uint32_t q_lo = sw128_desc_lo(smem_u32(smem + L::kQ + qs * L::kQTileBytes), 16);
        for (int j = 0; j < t.n; ++j, ++g) {
          const int b = g % SB, slot = g % RK;
          // Buffer b last held P(g - SB): PV(g - SB) must have read it.
          if (g >= SB && !mbar_wait(bar(kPVDone + b), ((g / SB) - 1) & 1, ctl)) { ok = false; break; }
          if (!mbar_wait(bar(kKFull + slot), (g / RK) & 1, ctl)) { ok = false; break; }
          const uint32_t kb = k_lo0 + (uint32_t)((slot * L::kTileBytes) >> 4);
          const uint32_t dS = tmem + (uint32_t)(b * kBN);
          // k steps of 32 bytes (16 bf16 or 32 e4m3) along each 128-byte span
#pragma unroll
          for (int kk = 0; kk < D * (FP8 ? 1 : 2) / 32; ++kk) {
            const uint32_t qoff = ((kk >> 2) * L::kQChunkBytes + (kk & 3) * 32) >> 4;
            const uint32_t koff = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
            if constexpr (FP8)
              mma_ss_lo_f8(dS, q_lo + qoff, kb + koff, dhi, id_s, kk > 0);
            else
              mma_ss_lo(dS, q_lo + qoff, kb + koff, dhi, id_s, kk > 0);
          }
          if constexpr (XB) {
            // One more k step adds slope (j - kv0) with the sign of j - i
            // (Q' K'+ below the diagonal, Q' K'- above it).  A non-causal
            // tile on the diagonal holds both signs: its softmax adds the
            // whole bias itself.
            const int kv0 = key_tile_at<VARIANT>(t, j, p.causal) * kBN;
            if (p.causal || kv0 != t.qrel) {
              // 32-byte swizzle, K-major; A (Q') with an 8-row stride of 0
              // (one atom for all rows), B (K'+-) with 256 bytes.
              const uint32_t qx = sw128_desc_lo(smem_u32(smem + L::kQx + qs * L::kQxBytes), 16);
              const uint32_t kx = sw128_desc_lo(
                  smem_u32(smem + ((p.causal || kv0 < t.qrel) ? L::kKxPos : L::kKxNeg)), 16);
              mma_ss_lo2(dS, qx, sw32_desc_hi(0), kx, sw32_desc_hi(256), id_s, 1u);
            }
          }
          mma_commit(bar(kSFull + b));
          mma_commit(bar(kKEmpty + slot));
        }
        if (ok) mma_commit(bar(kQEmpty + qs));  // every S product of this item has read Q
      }
      // Before TMEM can be freed every issued MMA must have finished.
      mma_commit(bar(kDrainS));
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
      mbar_wait(bar(kDrainS), 0, drain);
    }
    __syncwarp();
  } else if (warp == kPVWarp) {
    // ============================ O += P V issuer ============================
    if (lane == 0) {
      // bf16 V: MN-major, the head dimension's two 64-column halves one
      // chunk apart (LBO); e4m3 V^T: K-major like K.
      const uint32_t v_lo0 = sw128_desc_lo(smem_u32(smem + L::kV), FP8 ? 16 : L::kChunkBytes);
      bool ok = true;
      int g = 0;
      for (int r = 0; ok; ++r) {
        const int w = item_of(r, total);
        if (w < 0) break;
        const int n = tile_of<VARLEN, VARIANT, kBN>(w, p, seqt).n;
        const int ob = r % OB;
        const uint32_t tOr = o_buf(r);
        for (int j = 0; j < n; ++j, ++g) {
          const int b = g % SB, slot = g % RV;
          if (!mbar_wait(bar(kPFull + b), (g / SB) & 1, ctl)) { ok = false; break; }
          // The first product of an item overwrites its O buffer: the epilogue
          // must have read that buffer's previous item (r - OB) out of TMEM.
          if (j == 0 && r >= OB && !mbar_wait(bar(kOEmpty + ob), ((r / OB) - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();  // P(g) was written to TMEM by the softmax threads
          if (!mbar_wait(bar(kVFull + slot), (g / RV) & 1, ctl)) { ok = false; break; }
          // B = V tile rows [16kk, 16kk+16): 16 rows x 128 B per k step; the
          // 64-column halves of the head dimension are one chunk apart (LBO).
          const uint32_t vb = v_lo0 + (uint32_t)((slot * L::kTileBytes) >> 4);
          const uint32_t aP = tmem + (uint32_t)(b * kBN);
          const uint32_t acc0 = j > 0 ? 1u : 0u;
          if constexpr (FP8) {
            // 32 keys per step: 8 columns of P (four e4m3 per column), 32 bytes of each V^T row
#pragma unroll
            for (int kk = 0; kk < kBN / 32; ++kk)
              mma_ts_lo_f8(tOr, aP + kk * 8, vb + ((kk * 32) >> 4), dhi, id_pv, kk > 0 ? 1u : acc0);
          } else {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              mma_ts_lo(tOr, aP + kk * 8, vb + ((kk * 16 * 128) >> 4), dhi, id_pv,
                        kk > 0 ? 1u : acc0);
          }
          mma_commit(bar(kVEmpty + slot));
          mma_commit(bar(kPVDone + b));
          if (j == n - 1) mma_commit(bar(kOFull + ob));
        }
      }
      mma_commit(bar(kDrainPV));
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
      mbar_wait(bar(kDrainPV), 0, drain);
    }
    __syncwarp();
  } else if (warp < kProducerWarp) {
    // ============================ softmax warps ============================
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int row = warp * 32 + lane;               // row within the tile (= TMEM lane)
    bool ok = true;
    int g = 0;
    for (int r = 0; ok; ++r) {
      const int w = item_of(r, total);
      if (w < 0) break;
      const Tile t = tile_of<VARLEN, VARIANT, kBN>(w, p, seqt);
      const uint32_t tOm = o_buf(r) + lane_base;  // this item's O buffer
      const int q0 = t.qrel, q_row = q0 + row;  // indices within the sequence
      float m = -INFINITY, l = 0.f;   // running max (log2 domain) and sum of the row
      // ALiBi: this head's slope in log2 units.  At head_dim <= 128 the
      // tensor core has added its per-key part to S and each row adds a
      // constant per tile; otherwise the scores are biased and scaled in
      // place, so the passes below use a unit scale.
      float alibi_l2 = 0.f, sl2 = p.sl2, alibi_s = 0.f;
      if constexpr (VARIANT == kWindowAlibi) {
        alibi_l2 = p.alibi_slopes[t.zq % p.n_q_heads] * kLog2e;
        if constexpr (XB)
          alibi_s = alibi_l2 / p.sl2;  // the slope in units of S
        else
          sl2 = 1.f;
      }
      // FP8: the scores carry the Q block's scale (here) and the K block's
      // (per key tile, below).
      float q_scale = 1.f;
      if constexpr (FP8) q_scale = p.q_scales[(size_t)t.zq * p.n_q_tiles + t.tile0 + t.qrel / kBM];
      for (int j = 0; j < t.n; ++j, ++g) {
        const int b = g % SB;
        if constexpr (FP8)
          sl2 = p.sl2 * q_scale * p.k_scales[(size_t)t.zk * p.n_q_tiles + t.tile0 + t.j0 + j];
        if (!mbar_wait_warp(bar(kSFull + b), (g / SB) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tSm = tmem + (uint32_t)(b * kBN) + lane_base;
        // The whole S row: four 32-column loads in flight, one wait.
        float s[kBN];
        {
          uint32_t rr[kBN / 32][32];
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tSm + c * 32, rr[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(rr[c][i]);
        }
        const int kv0 = key_tile_at<VARIANT>(t, j, p.causal) * kBN;  // first key of the tile
        float c_row = 0.f;  // ALiBi (head_dim <= 128): the row's bias constant for this tile
        if constexpr (VARIANT != kPlain) {
          if constexpr (VARIANT == kWindowCap) {
            // This flavour requires softcap > 0 (cap_in2 != 0): with a zero
            // factor every r would be 1/2 and the softmax uniform.  The host
            // launches it only then (launch_prefill_t refuses otherwise).
            // s -> softcap * tanh(s * scale / softcap) with tanh = 1 - 2 r,
            // r = 1 / (2^v + 1), v = s * cap_in2: s keeps r, the max below
            // takes the smallest r and the exponent folds 1 - 2 r into its
            // FMA (softcap and log2 e are in sl2).  Masked scores get r = +inf.
            // (the multiply and the +1 on pairs: one instruction for two scores)
            const float2 ci = make_float2(p.cap_in2, p.cap_in2), one = make_float2(1.f, 1.f);
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
              const float2 v = mul2(make_float2(s[c], s[c + 1]), ci);
              const float2 e1 = add2(make_float2(ex2_approx(v.x), ex2_approx(v.y)), one);
              s[c] = rcp_approx(e1.x);
              s[c + 1] = rcp_approx(e1.y);
            }
          }
          if constexpr (VARIANT == kWindowAlibi) {
            const float dist0 = static_cast<float>(kv0 - q_row);  // key c is at j - i = dist0 + c
            if constexpr (XB) {
              // -slope |i - j| = -slope |i - kv0| +- slope (j - kv0): the
              // second term is in S already, the first is the row's constant.
              if (p.causal || kv0 != q0) {
                c_row = -alibi_l2 * fabsf(dist0);
              } else {
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                  s[c] = fmaf(-alibi_s, fabsf(dist0 + static_cast<float>(c)), s[c]);
              }
            } else {
              // s -> s scale log2 e - slope log2 e |i - j|
#pragma unroll
              for (int c = 0; c < kBN; ++c)
                s[c] = fmaf(s[c], p.sl2, -alibi_l2 * fabsf(dist0 + static_cast<float>(c)));
            }
          }
          const bool hi_edge = p.causal ? (kv0 + kBN - 1 > q0) : (kv0 + kBN > t.len);
          const bool lo_edge = p.window_left >= 0 && kv0 < q0 + kBM - 1 - p.window_left;
          if (hi_edge || lo_edge) {
            const int lim = !hi_edge ? kBN : p.causal ? (q_row - kv0) : (t.len - 1 - kv0);
            const int lo = lo_edge ? (q_row - p.window_left - kv0) : -1;  // first allowed column
            if constexpr (kChunkMask) {
              const int lim_w = (hi_edge && p.causal) ? lim - lane : lim;
              const int lo_w = lo_edge ? lo + (31 - lane) : -1;
#pragma unroll
              for (int ch = 0; ch < kBN / 32; ++ch)
                if (ch * 32 + 31 > lim_w || ch * 32 < lo_w)
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    const int c = ch * 32 + i;
                    if (c > lim || c < lo) s[c] = VARIANT == kWindowCap ? INFINITY : -INFINITY;
                  }
            } else {
#pragma unroll
              for (int c = 0; c < kBN; ++c)
                if (c > lim || c < lo) s[c] = VARIANT == kWindowCap ? INFINITY : -INFINITY;
            }
          }
        } else if (p.causal ? (kv0 + kBN - 1 > q0) : (kv0 + kBN > t.len)) {
          const int lim = p.causal ? (q_row - kv0) : (t.len - 1 - kv0);  // last allowed column
          if constexpr (kChunkMask) {
            const int lim_w = p.causal ? lim - lane : lim;  // the warp's first row's limit
#pragma unroll
            for (int ch = 0; ch < kBN / 32; ++ch)
              if (ch * 32 + 31 > lim_w)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (ch * 32 + i > lim) s[ch * 32 + i] = -INFINITY;
          } else {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c > lim) s[c] = -INFINITY;
          }
        }
        // Row max: eight independent chains of 3-input max, then a small tree
        // (soft-capping: the smallest r, the largest tanh = 1 - 2 r).
        float mx;
        if constexpr (VARIANT == kWindowCap) {
          float mna[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mna[k] = fminf(s[k], s[k + 8]);
#pragma unroll
          for (int c = 16; c < kBN; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) mna[k] = fmin3(mna[k], s[c + k], s[c + 8 + k]);
          const float mn = fmin3(fmin3(mna[0], mna[1], mna[2]), fmin3(mna[3], mna[4], mna[5]),
                                 fminf(mna[6], mna[7]));
          mx = fmaf(-2.f, mn, 1.f);  // -inf when every score of the row is masked
        } else {
          float mxa[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mxa[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
          for (int c = 16; c < kBN; c += 16)
#pragma unroll
            for (int k = 0; k < 8; ++k) mxa[k] = fmax3(mxa[k], s[c + k], s[c + 8 + k]);
          mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]),
                     fmaxf(mxa[6], mxa[7]));
        }
        const float m_new = fmaxf(m, XB ? fmaf(mx, sl2, c_row) : mx * sl2);
        // Rescale only when some row of the warp gained more than 2^8; otherwise
        // keep the stale max for both l and O (exact either way).
        float corr = 1.f;
        bool rescale_o = false;
        if constexpr (VARIANT != kPlain && VARIANT != kFp8) {
          // A row that has seen no allowed key yet (its keys so far were all
          // outside its window) has O = 0 and l = 0: it takes the new max
          // without a rescale.
          if (m == -INFINITY) m = m_new;
        }
        if (j == 0) {
          m = m_new;  // O is written fresh by the item's first P V product
        } else if (__any_sync(0xffffffffu, m_new - m > kRescaleThreshold)) {
          // The rescale is warp-wide: a row still without an allowed key
          // (m = m_new = -inf, l = 0, O = 0) keeps corr = 1 rather than
          // exp2(-inf + inf).
          corr = (VARIANT != kPlain && m_new == -INFINITY) ? 1.f : ex2_approx(m - m_new);
          m = m_new;
          l *= corr;
          rescale_o = true;
        }
        // P = exp2(s * scale * log2e - m): packed FMA for the argument, MUFU ex2,
        // packed into bf16 pairs over the first 64 columns of the buffer; the row
        // sum uses four packed chains.
        // A row whose keys in this item's tiles so far were all outside its
        // window has m = -inf (all its P are 0): take 0 as its reference.
        const float m_ref = (VARIANT != kPlain && m == -INFINITY) ? 0.f : m;
        const float nm = XB ? c_row - m_ref : -m_ref;
        const float2 sl2v = make_float2(sl2, sl2), nmv = make_float2(nm, nm);
        // soft-capping: exponent sl2 (1 - 2 r) - m = -2 sl2 r + (sl2 - m)
        const float2 cap_a = make_float2(-2.f * sl2, -2.f * sl2), cap_b = make_float2(sl2 - m_ref, sl2 - m_ref);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          if constexpr (FP8) {
            // e4m3 P: four keys per 32-bit column, key k in byte k % 4
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 x0 = fma2(make_float2(s[c * 32 + 4 * i], s[c * 32 + 4 * i + 1]), sl2v, nmv);
              const float2 x1 =
                  fma2(make_float2(s[c * 32 + 4 * i + 2], s[c * 32 + 4 * i + 3]), sl2v, nmv);
              const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
              const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
              rs[(2 * i) & 3] = add2(rs[(2 * i) & 3], p0);
              rs[(2 * i + 1) & 3] = add2(rs[(2 * i + 1) & 3], p1);
              pk[i] = e4m3x2_pack(p0.y, p0.x) | (e4m3x2_pack(p1.y, p1.x) << 16);
            }
            tmem_st8(tSm + c * 8, pk);
          } else {
            // Packed sequences: two stores of 16 keys (8 columns) each, which
            // keeps fewer registers live (8% faster there); the other
            // flavours measure faster with one store of 32 keys.
            constexpr int kPiece = VARLEN ? 8 : 16;  // packed columns per store
#pragma unroll
            for (int hh = 0; hh < 16 / kPiece; ++hh) {
              uint32_t pk[kPiece];
#pragma unroll
              for (int i = 0; i < kPiece; ++i) {
                const int k2 = c * 32 + hh * 2 * kPiece + 2 * i;
                const float2 x = VARIANT == kWindowCap
                                     ? fma2(make_float2(s[k2], s[k2 + 1]), cap_a, cap_b)
                                     : fma2(make_float2(s[k2], s[k2 + 1]), sl2v, nmv);
                const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rs[i & 3] = add2(rs[i & 3], pp);
                pk[i] = pack_bf16x2(pp.x, pp.y);
              }
              if constexpr (kPiece == 8)
                tmem_st8(tSm + c * 16 + hh * 8, pk);
              else
                tmem_st16(tSm + c * 16, pk);
            }
          }
        }
        const float2 rsum = add2(add2(rs[0], rs[1]), add2(rs[2], rs[3]));
        l += rsum.x + rsum.y;
        if (rescale_o) {
          // O must hold every P V product up to key tile j-1 before it is rescaled.
          const int bp = (g - 1) % SB;
          if (!mbar_wait_warp(bar(kPVDone + bp), ((g - 1) / SB) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tOm + c * 32, rr);
            tmem_wait_ld();
            const float2 cv = make_float2(corr, corr);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v =
                  mul2(make_float2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1])), cv);
              rr[2 * i] = __float_as_uint(v.x);
              rr[2 * i + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tOm + c * 32, rr);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kPFull + b));
      }
      if (!ok) break;
      // Row statistics to the epilogue warps (two slots, alternating items).
      const int ss = r & 1;
      if (r >= 2 && !mbar_wait_warp(bar(kStEmpty + ss), ((r >> 1) - 1) & 1, ctl)) { ok = false; break; }
      stats[ss * 128 + row] = make_float2(m, l);
      mbar_arrive(bar(kStFull + ss));
    }
  } else if (warp >= kEpiWarp0) {
    // ======================= epilogue: O = acc / l, LSE =======================
    // Warp w may access TMEM lanes [32 (w % 4), 32 (w % 4) + 32).
    // Each warp writes its 32 rows of O through a 4 KB staging box in shared
    // memory (32 rows x 32 floats, 128-byte swizzle: conflict-free row-wise
    // writes) and one TMA store per 32 columns, so the global writes are
    // whole lines and the load/store unit stays free for the softmax warps.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_q = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage = smem_u32(smem + L::kStage + quarter * 4096);
    const uint64_t pol_out = l2_policy_evict_first();  // O is not read again here
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = item_of(r, total);
      if (w < 0) break;
      const Tile t = tile_of<VARLEN, VARIANT, kBN>(w, p, seqt);
      const int ob = r % OB;
      const uint32_t tOm = o_buf(r) + lane_q;  // this item's O buffer
      if (!mbar_wait_warp(bar(kOFull + ob), (r / OB) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const int ss = r & 1;
      const int row0 = t.row0 + quarter * 32;  // tensor row of this warp's box
      // Rows of the box inside the sequence.  A padded batch's boxes end at
      // the tensor's end, where the copy clips; a packed sequence's last box
      // may reach into the next sequence, so it is written row by row.
      const int in_seq = t.len - (t.qrel + quarter * 32);
      // O is read kEC columns at a time (all of it for head_dim <= 128).
      constexpr int kEC = D > 128 ? 128 : D;
      const int d_out = FP8 ? p.d_out : D;  // O's columns in memory
      auto store_cols = [&](const uint32_t (&acc)[kEC / 32][32], int col0, float inv_l) {
        if constexpr (OBF16) {
          // bf16 O: 64 columns make one 128-byte row of the staging box.
          auto pk = [&](int c, int b) {  // columns b, b+1 of 32-column chunk c, as bf16x2
            return __uint_as_float(pack_bf16x2(__uint_as_float(acc[c][b]) * inv_l,
                                               __uint_as_float(acc[c][b + 1]) * inv_l));
          };
          if (!VARLEN || in_seq >= 32) {
#pragma unroll
            for (int c2 = 0; c2 < kEC / 64; ++c2) {
              if (FP8 && col0 + c2 * 64 >= d_out) break;
              if (lane == 0) bulk_wait_read_all();  // the previous box has left the buffer
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 8; ++i) {  // 8 columns per 16-byte piece
                const int c = 2 * c2 + (i >> 2), b = (i & 3) * 8;
                st_shared_v4(stage + lane * 128 + ((i ^ (lane & 7)) << 4),
                             make_float4(pk(c, b), pk(c, b + 2), pk(c, b + 4), pk(c, b + 6)));
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0 && row0 < N) {  // rows past the tensor's end are clipped by the copy
                tma_store_3d_hint(&tm_o, stage, col0 + c2 * 64, row0, t.zq, pol_out);
                bulk_commit_group();
              }
            }
          } else if (lane < in_seq) {
            uint16_t* orow = static_cast<uint16_t*>(p.o) +
                             ((size_t)t.zq * N + (size_t)(row0 + lane)) * d_out + col0;
#pragma unroll
            for (int c = 0; c < kEC / 32; ++c) {
              if (FP8 && col0 + c * 32 >= d_out) continue;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                reinterpret_cast<float4*>(orow + c * 32)[i] =
                    make_float4(pk(c, 8 * i), pk(c, 8 * i + 2), pk(c, 8 * i + 4), pk(c, 8 * i + 6));
            }
          }
          return;
        }
        if (!VARLEN || in_seq >= 32) {
#pragma unroll
          for (int c = 0; c < kEC / 32; ++c) {
            if (FP8 && col0 + c * 32 >= d_out) break;
            if (lane == 0) bulk_wait_read_all();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_shared_v4(stage + lane * 128 + ((i ^ (lane & 7)) << 4),
                           make_float4(__uint_as_float(acc[c][4 * i]) * inv_l,
                                       __uint_as_float(acc[c][4 * i + 1]) * inv_l,
                                       __uint_as_float(acc[c][4 * i + 2]) * inv_l,
                                       __uint_as_float(acc[c][4 * i + 3]) * inv_l));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && row0 < N) {  // rows past the tensor's end are clipped by the copy
              tma_store_3d_hint(&tm_o, stage, col0 + c * 32, row0, t.zq, pol_out);
              bulk_commit_group();
            }
          }
        } else if (lane < in_seq) {
          float* orow = static_cast<float*>(p.o) + ((size_t)t.zq * N + (size_t)(row0 + lane)) * d_out + col0;
#pragma unroll
          for (int c = 0; c < kEC / 32; ++c)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (FP8 && col0 + c * 32 >= d_out) continue;
              reinterpret_cast<float4*>(orow + c * 32)[i] =
                  make_float4(__uint_as_float(acc[c][4 * i]) * inv_l,
                              __uint_as_float(acc[c][4 * i + 1]) * inv_l,
                              __uint_as_float(acc[c][4 * i + 2]) * inv_l,
                              __uint_as_float(acc[c][4 * i + 3]) * inv_l);
            }
        }
      };
      float2 ml;
      if constexpr (D <= 128) {
        uint32_t acc[kEC / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tOm + c * 32, acc[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kOEmpty + ob));  // this O buffer may now take item r + OB
        if (!mbar_wait_warp(bar(kStFull + ss), (r >> 1) & 1, ctl)) { ok = false; break; }
        ml = stats[ss * 128 + row];
        mbar_arrive(bar(kStEmpty + ss));
        store_cols(acc, 0, (FP8 ? p.v_scales[t.zk] : 1.f) / ml.y);  // FP8: V's per-head scale
      } else {
        // head_dim 256: the row statistics first, then O in two halves; O is
        // released once its last half has been read.
        if (!mbar_wait_warp(bar(kStFull + ss), (r >> 1) & 1, ctl)) { ok = false; break; }
        ml = stats[ss * 128 + row];
        mbar_arrive(bar(kStEmpty + ss));
        const float inv_l = 1.f / ml.y;
#pragma unroll 1
        for (int h = 0; h < D / kEC; ++h) {
          uint32_t acc[kEC / 32][32];
#pragma unroll
          for (int c = 0; c < kEC / 32; ++c) tmem_ld32(tOm + h * kEC + c * 32, acc[c]);
          tmem_wait_ld();
          if (h == D / kEC - 1) {
            tc_fence_before();
            mbar_arrive(bar(kOEmpty + ob));
          }
          store_cols(acc, h * kEC, inv_l);
        }
      }
      if (t.qrel + row < t.len && t.row0 + row < N)
        p.lse[(size_t)t.zq * N + t.row0 + row] = (ml.x + __log2f(ml.y)) * kLn2;
    }
    if (lane == 0) bulk_wait_all();  // O is in global memory before the CTA exits
    __syncwarp();
  }

  // ---- teardown: every TMEM reader and both MMA drains are done ----
  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// (rows, planes) bf16 tensor of shape (planes, rows, D): box = 64 x box_rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int rows, int planes, int box_rows = 128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 (planes, rows, inner): box = 128 x 128 x 1 (128-byte rows), 128-byte swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, int inner, int rows, int planes) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)inner, (cuuint64_t)inner * (cuuint64_t)rows};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output (planes, rows, D), fp32 (box 32 x 32 x 1) or bf16 (box 64 x 32 x 1):
// 128-byte rows, 128-byte swizzle.
bool make_out_map(CUtensorMap* m, void* base, int D, int rows, int planes, bool bf16 = false) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t esz = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)D * esz, (cuuint64_t)D * esz * (cuuint64_t)rows};
  cuuint32_t box[3] = {bf16 ? 64u : 32u, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base,
             dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool VARLEN, int VARIANT, bool OBF16 = false>
cudaError_t launch_prefill_t(const PrefillArgs& a, const LaunchCtx& ctx) {
  constexpr bool FP8 = VARIANT == kFp8;
  using L = PrefillSmem<D, VARLEN, FP8 ? 1 : 2, VARIANT == kWindowAlibi && D <= 128>;
  // The soft-cap flavour drops the factor's zero test from its hot loop.
  if (VARIANT == kWindowCap && !(a.softcap > 0.f)) return cudaErrorInvalidValue;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, VARLEN, VARIANT, OBF16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  CUtensorMap mq, mk, mv, mo;
  // FP8 at head_dim 64 runs this 128-column kernel: the maps cover the real
  // 64 columns (rows of V^T) and the 128-wide boxes read zeros beyond them.
  const int d_io = FP8 ? a.head_dim : D;
  if (FP8) {
    // Q, K (planes, rows, d_io) and V transposed (planes, d_io, rows), e4m3
    if (!make_map_u8(&mq, a.q, d_io, a.seqlen, a.batch * a.n_q_heads) ||
        !make_map_u8(&mk, a.k, d_io, a.seqlen, a.batch * a.n_kv_heads) ||
        !make_map_u8(&mv, a.v, a.seqlen, d_io, a.batch * a.n_kv_heads))
      return cudaErrorInvalidValue;
  } else if (!make_map(&mq, a.q, D, a.seqlen, a.batch * a.n_q_heads) ||
             !make_map(&mk, a.k, D, a.seqlen, a.batch * a.n_kv_heads, key_tile<D>()) ||
             !make_map(&mv, a.v, D, a.seqlen, a.batch * a.n_kv_heads, key_tile<D>())) {
    return cudaErrorInvalidValue;
  }
  if (!make_out_map(&mo, a.o, d_io, a.seqlen, a.batch * a.n_q_heads, OBF16))
    return cudaErrorInvalidValue;
  PrefillParams pp;
  pp.o = a.o;
  pp.lse = a.lse;
  pp.batch = a.batch;
  pp.n_q_heads = a.n_q_heads;
  pp.n_kv_heads = a.n_kv_heads;
  pp.seqlen = a.seqlen;
  pp.sl2 = a.softcap > 0.f ? a.softcap * kLog2e : a.scale * kLog2e;
  pp.causal = a.causal;
  pp.window_left = a.window_left;
  pp.cap_in2 = a.softcap > 0.f ? 2.f * kLog2e * a.scale / a.softcap : 0.f;
  pp.alibi_slopes = a.alibi_slopes;
  pp.q_scales = a.q_scales;
  pp.k_scales = a.k_scales;
  pp.v_scales = a.v_scales;
  pp.d_out = d_io;
  // Padded: query tiles per sequence.  Packed: the columns of the FP8 scale
  // arrays (every sequence's tiles, at most ceil(total / 128) + num_seqs).
  pp.n_q_tiles = (a.seqlen + kBM - 1) / kBM + (VARLEN ? a.num_seqs : 0);
  pp.total_tiles = pp.n_q_tiles * a.batch * a.n_q_heads;
  pp.group_planes = a.batch * a.n_q_heads;  // one group: longest first over everything
  {
    // When the launch's K and V exceed 96 MB (L2 holds about 126 MB, and Q
    // and O stream through it too), group whole kv heads so that each group's
    // K and V take about 24 MB.
    const long long kv_plane = 2LL * a.seqlen * D * (FP8 ? 1 : 2);
    const long long kv_total = kv_plane * a.batch * a.n_kv_heads;
    if (VARIANT == kPlain && !VARLEN && kv_total > (96LL << 20)) {
      const int kvg = (int)std::max(1LL, (24LL << 20) / kv_plane);
      pp.group_planes = std::min(kvg * (a.n_q_heads / a.n_kv_heads), a.batch * a.n_q_heads);
    }
  }
  pp.cu_seqlens = a.cu_seqlens;
  pp.num_seqs = a.num_seqs;
  pp.seq_base = a.seq_base;
  pp.err_word = ctx.err_word;
  pp.timeout_ns = ctx.timeout_ns;
  // Persistent: one CTA per SM (shared memory and TMEM admit one), each
  // walking its share of the work list.  Packed sequences: the item count is
  // on the device, so every SM gets a CTA (those without items exit at once).
  const int sms = std::max(ctx.num_sms, 1);
  const unsigned grid = (unsigned)(VARLEN ? sms : std::min(pp.total_tiles, sms));
  prefill_kernel<D, VARLEN, VARIANT, OBF16><<<grid, kThreads, L::kAlloc, ctx.stream>>>(mq, mk, mv, mo,
                                                                                        pp);
  return cudaGetLastError();
}

}  // namespace

template <int D, bool VARLEN, bool OBF16>
cudaError_t launch_prefill_flavour(const PrefillArgs& a, const LaunchCtx& ctx) {
  if (a.alibi_slopes) return launch_prefill_t<D, VARLEN, kWindowAlibi, OBF16>(a, ctx);
  if (a.softcap > 0.f) return launch_prefill_t<D, VARLEN, kWindowCap, OBF16>(a, ctx);
  if (a.window_left >= 0) return launch_prefill_t<D, VARLEN, kWindow, OBF16>(a, ctx);
  return launch_prefill_t<D, VARLEN, kPlain, OBF16>(a, ctx);
}

template <int D, bool VARLEN>
cudaError_t launch_prefill_cap(const PrefillArgs& a, const LaunchCtx& ctx) {
  return a.o_bf16 ? launch_prefill_flavour<D, VARLEN, true>(a, ctx)
                  : launch_prefill_flavour<D, VARLEN, false>(a, ctx);
}

cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtx& ctx) {
  if (a.fp8) {
    if ((a.head_dim != 128 && a.head_dim != 64) || a.o_bf16) return cudaErrorInvalidValue;
    return a.cu_seqlens ? launch_prefill_t<128, true, kFp8>(a, ctx)
                        : launch_prefill_t<128, false, kFp8>(a, ctx);
  }
  const bool varlen = a.cu_seqlens != nullptr;
  if (a.head_dim == 256)
    return varlen ? launch_prefill_cap<256, true>(a, ctx) : launch_prefill_cap<256, false>(a, ctx);
  if (a.head_dim == 128)
    return varlen ? launch_prefill_cap<128, true>(a, ctx) : launch_prefill_cap<128, false>(a, ctx);
  return varlen ? launch_prefill_cap<64, true>(a, ctx) : launch_prefill_cap<64, false>(a, ctx);
}

}  // namespace attn
