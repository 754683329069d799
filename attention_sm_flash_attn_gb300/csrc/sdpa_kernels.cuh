// sdpa_kernels.cuh -- fused scaled-dot-product attention kernels for sm_103a.
//
// What is computed (the unfused "matmul + softmax + matmul" of the page
// "fix: add head_dim=256 to fused SDPA full attention kernel", section
// "Benchmark: fused vs unfused SDPA for head_dim=256", done tile by tile so the
// [heads, Lq, Lk] score matrix never exists):
//
//   for query row i of head h (kv head g = h / G, G = Hq / Hkv), position
//   p = Lk - Lq + i (bottom-right aligned), visible keys j with
//   (!causal || j <= p) && (window == 0 || p - j < window):
//     out[h, i] = sum_j softmax_j(scale * q_i . k_j) v_j
//
// One CTA owns 128 query rows (one tcgen05 M=128 tile; 256 rows per CTA pair
// in the 2-SM variants) and walks a list of key tiles.  Warp roles (384
// threads; the head-dim-split pairs add four exchange warps, see Cfg):
//   warps 0-7  softmax + epilogue: two threads per row / TMEM lane, warps q
//              and q+4 owning the two halves of the key (and O) columns
//   warp  8    TMA producer: Q, then K and V sub-tiles into a ring
//   warp  9    TMEM allocator and tcgen05.mma issuer
//   warps 10-11 idle (they complete the third warpgroup of the register split)
// Per key tile j:  S_j = Q K_j^T (tcgen05, fp32 in TMEM)
//                  softmax warps: tcgen05.ld S_j, mask, online max/sum (log2
//                  domain, lazy rescale), P_j (fp16/bf16) to tensor memory
//                  over S_j, or to shared memory (kDuoQ and the pairs)
//                  O += P_j V_j  (tcgen05, fp32 in TMEM)
// Whole key tiles outside the causal/window band are never visited.  With
// BIAS, an additive bias (a mask array) is added to the scaled scores.
//
// Modes:
//  * prefill: 128 (or 256) consecutive query rows of one head; either the
//    whole visible key range (final output), one contiguous share of it (fp32
//    partials merged by the combine kernel), or, in the persistent schedule,
//    a sequence of pieces of several query tiles with suffix pieces merged by
//    the unit that owns the tile's prefix;
//  * decode (Lq <= 8): the 128 rows are 16 query heads x 8 slots of one kv
//    head; query row i goes to slot (p_i mod 8), so the same row always lands
//    on the same TMEM lane whatever Lq is.  Key tiles are dealt round-robin
//    over a fixed number of splits, so the arithmetic one row sees does not
//    depend on how many query rows share the call ("fix: Gemma 4 MTP never
//    engages on CUDA (GB10)", sections "Proposed Solution" and "Acceptance
//    Criteria": a verify row must be byte-identical to the single-row call).
//  * PAIR (head_dim 512, kPairX / kPairXD): a 2-CTA cluster splits the head
//    dimension; each CTA forms its half of the scores, the halves are swapped
//    through distributed shared memory and summed (both CTAs add the same two
//    fp32 numbers, so both run an identical softmax), then each CTA
//    accumulates its half of O.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace gbsdpa {

// Barrier that signals "S buffer `buf` (0 or 1) holds a finished Q.K^T product".
__host__ __device__ constexpr int sfull_bar(int buf) { return 17 + buf; }

// Device status codes (bit pattern identifies the wait that gave up).
enum : int {
  kDevOk = 0,
  kDevTimeoutQ = 0x100,
  kDevTimeoutKvFull = 0x101,
  kDevTimeoutKvEmpty = 0x102,
  kDevTimeoutSFull = 0x103,
  kDevTimeoutSEmpty = 0x104,
  kDevTimeoutPFull = 0x105,
  kDevTimeoutPvDone = 0x106,
  kDevTimeoutXFull = 0x107,
  kDevTimeoutXFree = 0x108,
  kDevTimeoutDrain = 0x109,
  kDevTimeoutPair = 0x10a,  // a prefix unit waited too long for a suffix piece's partials
  kDevMisaligned = 0x10b,
  kDevBadCluster = 0x10c,  // a 2-CTA variant was launched without a cluster of 2
  kDevBadGrid = 0x10d,     // a decode CTA found no work item of the call (grid too large)
};

struct AttnParams {
  CUtensorMap tm_q;  // (D, Lq, B*Hq) box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;  // (D, Lk, B*Hkv) box (64, BN, 1)
  CUtensorMap tm_v;  // (D, Lk, B*Hkv) box (64, 32, 1)
  const uint16_t* q;
  uint16_t* out;
  float* part_o;   // [n_splits][B*Hq*Lq][D]
  float* part_ml;  // [n_splits][B*Hq*Lq][2]  (running max in log2 units, sum)
  int* status;
  int B, Hq, Hkv, G, Lq, Lk, D;  // D: head dim of V and the output
  int Dqk;                       // head dim of Q and K
  int causal, window;
  float c;        // scale * log2(e)
  int decode;     // 0 = prefill, 1 = decode
  int n_qtiles;   // prefill: query tiles per head (ceil(Lq / rows of a tile))
  // 2-SM variants: 1 = a CTA pair owns 128 query rows of two query heads of one
  // kv head (CTA `rank` takes head 2 * pair + rank), 0 = 256 consecutive rows
  // of one head (CTA `rank` takes rows 128 * rank ..).
  int hpair;
  int n_splits;   // prefill: 1 => final output written directly; decode: fixed split count
  int n_hb;       // decode: query-head blocks of 16 per kv head
  // kDecode: the n_splits splits of a (batch, kv head, head block) group are
  // dec_nc clusters of dec_cs CTAs; a cluster merges its splits through
  // distributed shared memory and writes the output (dec_nc == 1) or one fp32
  // partial per cluster for the combine kernel (dec_nc > 1).
  int dec_cs, dec_nc;
  int write_partial;
  // Self-test only (always 0 on the normal entry points): 1 = withhold the
  // "query tile ready" signal, so the MMA issuer's bounded wait runs out and the
  // kernel reports a device timeout instead of computing; 2 = suffix pieces of
  // the persistent schedule never publish their flags, so the prefix units'
  // bounded waits run out.
  int withhold_q;
  // K/V rows: key j is row j of its (b, kv head) plane, or, for a ring buffer of
  // kv_ring rows (a multiple of 128), row j mod kv_ring.
  int kv_ring;
  // Persistent prefill (SINGLE and DUO variants): `n_units` resident CTAs (CTA
  // pairs for DUO) walk the query tiles ("items") in waves, then share out the
  // leftover partial wave so that every unit gets about the same number of key
  // tiles.  A leftover item is cut into a prefix, finished by one unit, and a
  // suffix that other units compute in pieces; each piece leaves fp32 partials
  // in its slot of sk_o / sk_ml and sets its flag to `epoch`, and the prefix
  // unit merges them in key order.
  int persistent;
  int n_units;
  int tail_L;        // prefix length (key tiles) of the leftover items
  int tail_US;       // suffix units
  long long tail_SS; // suffix key tiles in all
  float* sk_o;                 // [n_units][2][128][256]  (slot, rank, row, column)
  float* sk_ml;                // [n_units][2][128][2]
  unsigned long long* sk_flag; // [n_units][2]
  unsigned long long epoch;
  // Additive bias (a mask array), or null: entry (b, h, i, j) at
  // bias[b * bias_sb + h * bias_sh + i * bias_sq + j] (elements, q's dtype; a
  // stride of 0 broadcasts), added to the scaled score of query row i and key j.
  // bias_vec = 1: base and strides are 16-byte multiples, so a row is read in
  // 8-element vectors.
  const uint16_t* bias;
  long long bias_sb, bias_sh, bias_sq;
  int bias_vec;
};

// Kernel variants.
//   kSingle: one CTA per 128 query rows: prefill at head_dim 192 (and Q/K 192
//            with V 256), and prefill with a window under 256 keys.
//   kDuo:    head_dim 256 prefill with 2-SM MMAs (cta_group::2): a 2-CTA
//            cluster owns 256 query rows; each CTA loads half of every K and V
//            tile, which halves the bytes each SM stages per FLOP.
//   kDuoQ:   the 2-SM variant with Q in tensor memory (Q.K^T reads its A
//            operand from TMEM), one S buffer and P in shared memory.
//   kDecode: decode (Lq <= 8) at head_dim <= 256: one CTA per split over
//            64-key tiles; the splits of a (batch, kv head, head block) form a
//            thread-block cluster and merge their partials through distributed
//            shared memory at the end, so one launch writes the output.
//   kPairX:  head_dim 512: a 2-CTA cluster splits the head dimension and swaps
//            partial scores through distributed shared memory.  Four exchange
//            warps read this CTA's partial scores from tensor memory and send
//            them to the peer (up to two tiles ahead); eight softmax warps add
//            the two halves from shared memory.  Q in tensor memory, P through
//            shared memory.
//   kPairXD: kPairX for decode (Lq <= 8): an 8-slot K/V ring and one exchange
//            slot instead of a 5-slot ring and two, which keeps more of the
//            K/V stream in flight (the prefill kernel measured slower with it).
// (Value 1 belonged to an earlier head_dim-512 pair that the exchange warps
// replaced; the numbers of the others are kept.)
enum Mode : int { kSingle = 0, kDuo = 2, kDuoQ = 3, kDecode = 4, kPairX = 5, kPairXD = 6 };
constexpr int kNumModes = 7;

template <bool BF16, int MODE, int HD = 256, int HDV = HD, bool BIAS = false>
struct Cfg {
  static constexpr bool PX = MODE == kPairX || MODE == kPairXD;
  static constexpr bool PXD = MODE == kPairXD;
  static constexpr bool PAIR = PX;  // head dim split over a CTA pair
  static constexpr bool DUO = MODE == kDuo || MODE == kDuoQ;
  static constexpr bool DEC = MODE == kDecode;
  static constexpr int BM = 128;                   // query rows per CTA
  static constexpr int DH = HD;                    // Q/K head-dim columns owned by one CTA
  static constexpr int DV = HDV;                   // V (and output) head-dim columns
  static constexpr int BN = (PAIR || DEC) ? 64 : 128;  // keys per tile
  static constexpr int HB = BN / 2;                // key columns per softmax thread
  static constexpr int NSLOT = (PX && !PXD) ? 5 : 8;
  static constexpr int SLOT = 16384;
  // K per CTA and tile: DUO holds 64 of the 128 keys, the others all BN keys.
  static constexpr int KROWS = DUO ? 64 : BN;      // rows of a K box
  // 64-column K boxes per slot: as many as fit (two of 64 rows, one of 128),
  // fewer when the head dim's box count does not divide by that (192 = 3 boxes
  // of 64 rows go one to a slot).
  static constexpr int KBOX_FIT = SLOT / (KROWS * 128);
  static constexpr int KBOX = (DH / 64) % KBOX_FIT == 0 ? KBOX_FIT : 1;
  static constexpr int KSUB = DH / 64 / KBOX;      // K slots per tile
  // V per CTA and tile: DUO holds 128 of the 256 head-dim columns for all keys,
  // in slots of 64 keys x 128 columns; the others hold slots of 32 keys x 256.
  static constexpr int VROWS = DUO ? 64 : 32;      // keys per V slot (= rows of a V box)
  static constexpr int VBOX = (DUO ? DV / 2 : DV) / 64;  // 64-column V boxes per slot
  static constexpr int VSUB = BN / VROWS;          // V slots per tile
  static constexpr int V_LBO = VROWS * 128;        // bytes between 64-column V boxes
  // Bytes one CTA loads into a ring slot (a V slot is not full below head_dim 256).
  static constexpr int K_SLOT_BYTES = KBOX * KROWS * 128;
  static constexpr int V_SLOT_BYTES = VBOX * V_LBO;
  // Q in tensor memory (kDuoQ, kPairX): Q.K^T reads its A operand from TMEM.
  // P through shared memory (PSM: kDuoQ, kPairX): P.V reads its A operand from
  // a swizzled shared-memory buffer, and an S buffer is released by its own
  // barrier (SFREE) once its scores have been read.  The other variants keep Q
  // in shared memory and P in TMEM over the S buffer it came from.
  static constexpr bool QTM = MODE == kDuoQ || PX;
  static constexpr bool PSM = MODE == kDuoQ || PX;
  static constexpr bool SFREE = PSM;
  // Epilogue through shared memory (STAGE, kDuoQ, in its P buffer): each warp
  // stages 32 rows x 64 columns of the output and writes whole 128-byte lines.
  // (The same staging in the other 2-SM kernel, in a buffer of its own,
  // measured no faster on the sliding-window prefill, so it keeps direct
  // stores and its smaller shared-memory footprint.)
  static constexpr bool STAGE = MODE == kDuoQ;
  // Shared memory.  Most variants: Q tile, ring, [P], barriers, row swap
  // area, iterators.  kPairX: ring (5 slots), X and XS (two slots each), P,
  // barriers, row swap area, iterators.  kPairXD: ring (8 slots), X, XS, P,
  // 16 KB spare, barriers, ...  The pairs stage the query tile over XS (and
  // P and the spare) before it is copied to TMEM: those are first written
  // after the first Q.K^T, which follows that copy.
  static constexpr int RING_OFF = PX ? 0 : 65536;
  static constexpr int RING_END = RING_OFF + NSLOT * SLOT;
  static constexpr int X_SLOTS = (PX && !PXD) ? 2 : 1;  // exchange slots (X and XS)
  static constexpr int P_BYTES = PSM ? BM * BN * 2 : 0;
  static constexpr int X_BYTES = PAIR ? BM * BN * 4 : 0;      // one slot
  static constexpr int X_OFF = PX ? RING_END : RING_END + P_BYTES;  // peer's partial scores
  static constexpr int XS_OFF = X_OFF + X_SLOTS * X_BYTES;    // own partial scores to send
  static constexpr int P_OFF = PX ? XS_OFF + X_SLOTS * X_BYTES : RING_END;
  static constexpr int Q_OFF = PX ? XS_OFF : 0;
  static constexpr int BAR_OFF =
      PX ? P_OFF + P_BYTES + (PXD ? 16384 : 0) : XS_OFF + X_SLOTS * X_BYTES;
  static constexpr int RED_OFF = BAR_OFF + 256;      // [2 parity][2 half][128 rows] floats
  static constexpr int RED_BYTES = 2048;
  // Piece iterators: softmax warps (state + 2 pieces), producer and MMA issuer
  // (state + 1 piece each), 256 bytes apiece.
  static constexpr int ITER_OFF = RED_OFF + RED_BYTES;
  static constexpr int SMEM_BYTES = ITER_OFF + 768;
  static constexpr int S_COL = 256;  // TMEM: O in columns [0,256), S buffers after it
  // S buffers: kDuoQ has one, the others two.
  static constexpr int NSBUF = MODE == kDuoQ ? 1 : 2;
  // Q.K^T products the MMA issuer keeps ahead of P.V (the pair runs two tiles
  // ahead while the exchange warps swap partial scores with the peer).
  static constexpr int S_AHEAD = PX ? 2 : 1;
  static constexpr int Q_COL = S_COL + NSBUF * BN;   // Q (QTM): DH/2 columns
  // Warps 0-7 softmax (warpgroups 0, 1).  kPairX: 8-11 exchange (warpgroup 2),
  // 12 producer, 13 MMA, 14-15 idle (warpgroup 3).  Others: 8 producer, 9 MMA,
  // 10-11 idle (warpgroup 2).
  static constexpr int NTHREADS = PX ? 512 : 384;
  static constexpr int kLaunchRegs = PX ? 128 : 168;  // 64K registers / threads, rounded down to 8
  // Registers a thread after the split; the sum stays within the launch
  // allotment of NTHREADS x kLaunchRegs.
  static constexpr int kRegsSoftmax = PX ? 160 : 208;
  static constexpr int kRegsExchange = 104;
  static constexpr int kRegsOther = PX ? 80 : 88;
  static_assert(256 * kRegsSoftmax + (PX ? 128 * kRegsExchange : 0) + 128 * kRegsOther <=
                    NTHREADS * kLaunchRegs,
                "register split");
  static constexpr int kExchangeWarp = 8;  // kPairX: first exchange warp
  static constexpr int kProducerWarp = PX ? 12 : 8;
  static constexpr int kMmaWarp = PX ? 13 : 9;
  static constexpr int MMA_M = DUO ? 256 : 128;
  static constexpr uint32_t IDESC_QK = ptx::idesc_f16(MMA_M, BN, BF16, false, false);
  // P.V: N = DV (the 2-SM variant's B operand is two DV/2-column halves).
  static constexpr uint32_t IDESC_PV = ptx::idesc_f16(MMA_M, DV, BF16, false, true);
  static constexpr int Q_BYTES = BM * DH * 2;  // one CTA's query tile
  // Arrivals completing P-full on the MMA CTA: one per softmax warp of each CTA
  // whose P rows the MMA reads.
  static constexpr int kPFullArrivals = DUO ? 16 : 8;
  static_assert(S_COL + NSBUF * BN + (QTM ? DH / 2 : 0) <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  // Every region the kernel addresses lies inside the window it is launched with.
  static_assert(RED_OFF + RED_BYTES <= ITER_OFF && ITER_OFF + 768 <= SMEM_BYTES &&
                    P_OFF + P_BYTES <= (PX ? BAR_OFF : X_OFF) &&
                    XS_OFF + X_SLOTS * X_BYTES <= (PX ? P_OFF : BAR_OFF),
                "shared-memory regions overlap");
  static_assert(!PX || Q_OFF + Q_BYTES <= BAR_OFF, "query staging over XS, P and the spare");
  static_assert(!STAGE || (P_BYTES >= 8 * 4096 && DV == 256 && !PAIR),
                "the staged epilogue: 8 warps x 32 rows x 64 columns in the P buffer");
  static_assert(KSUB * KBOX * 64 == DH && VSUB * VROWS == BN, "tile decomposition");
  static_assert(VBOX * 64 == (DUO ? DV / 2 : DV) && V_SLOT_BYTES <= SLOT && K_SLOT_BYTES <= SLOT,
                "K/V slot layout");

  static_assert((PX ? Q_BYTES <= 2 * X_BYTES : Q_BYTES <= RING_OFF) &&
                    (!PAIR || (DH == 256 && DV == 256)) && DV <= S_COL,
                "query tile / pair head dim / O columns");
};

// Barrier slots inside the barrier area.
enum {
  kBarQ = 0,
  kBarKvFull = 1,    // + slot (8 slots max)
  kBarKvEmpty = 9,   // + slot
  kBarSFull = 17,    // + buf
  kBarQFree = 19,    // the last S of a piece has completed: Q may be reloaded
  kBarOFree = 20,    // the epilogue has read O: the next piece may overwrite it
  kBarPFull = 21,
  kBarPvDone = 22,
  kBarXFull = 23,
  kBarXFree = 24,
  kBarDrain = 25,
  kBarSFree = 26,    // Q in TMEM: the softmax has read the (single) S buffer
  kNumBars = 30,     // 27..29: kPairX exchange barriers (below)
};
static_assert(kNumBars * 8 <= 240, "barriers end below the TMEM slot and abort flag");
static_assert(sfull_bar(0) == kBarSFull && sfull_bar(1) == kBarSFull + 1, "S-full barriers");

// The pairs' exchange barriers, per exchange slot x (NX = 2 slots: kPairX,
// whose 5-slot ring leaves the ring barriers of slots 5..7 free; NX = 1:
// kPairXD, 8 ring slots) and S buffer b:
//   xfull   the peer's partial scores landed in our X slot (1 arrival + bytes)
//   xfree   the peer's softmax warps have read our block from its X slot (8)
//   sfree   our exchange warps have read S buffer b (4)
//   xsready our exchange warps have staged our partial scores in XS slot (4)
//   xsfree  our softmax warps have read XS slot (8)
__host__ __device__ constexpr int xfull_bar(int x) { return x ? 6 : kBarXFull; }
__host__ __device__ constexpr int xfree_bar(int x) { return x ? 7 : kBarXFree; }
template <int NX>
__host__ __device__ constexpr int sfree_bar(int b) { return b ? (NX == 2 ? 8 : 27) : kBarSFree; }
template <int NX>
__host__ __device__ constexpr int xsready_bar(int x) { return NX == 2 ? 14 + x : 28; }
template <int NX>
__host__ __device__ constexpr int xsfree_bar(int x) { return NX == 2 ? (x ? 27 : 16) : 29; }

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

// Largest decode cluster (CTAs); 16 is the non-portable cluster size.
constexpr int kMaxDecodeClusterCtas = 16;


// Bounded mbarrier wait.  Gives up after kTimeoutNs (or when another role of
// this CTA already gave up), records `code` in the device status word and
// returns false.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status, int code) {
  if (kCluster ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
    return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t n = 1; n < (1u << 30); ++n) {
    if (kCluster ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
      return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > kTimeoutNs) break;
    }
  }
  *abort_flag = 1;
  atomicCAS(status, 0, code);
  return false;
}

struct Work {
  int b, hkv, h0;      // batch, kv head, first query head of the CTA
  int split;
  int m0;              // prefill: first query row
  int pmin, pmax;      // positions spanned by the CTA's rows
  int t_begin, t_step, t_count;
};

// Query heads per prefill item and query rows per tile.  A 2-SM pair (QROWS
// 256) owns either 256 consecutive rows of one head or, with p.hpair, 128 rows
// of two heads of the same kv head; one CTA owns 128 rows of one head.
template <int QROWS>
__device__ __forceinline__ int item_heads(const AttnParams& p) {
  return (QROWS == 256 && p.hpair) ? 2 : 1;
}
template <int QROWS>
__device__ __forceinline__ int tile_rows(const AttnParams& p) {
  return (QROWS == 256 && !p.hpair) ? 256 : 128;
}

// Work of one CTA.  Prefill items walk (query heads within their group, split,
// kv head, batch, query tile) with the longest causal query tiles first; see
// item_heads / tile_rows for what an item of a 2-SM pair covers.  Decode items
// walk (head block, split, kv head, batch).
template <int BN, int QROWS>
__device__ __forceinline__ Work make_work(const AttnParams& p, int item, int rank) {
  Work w;
  int lo, hi;
  if (!p.decode) {
    const int ih = item_heads<QROWS>(p), rows = tile_rows<QROWS>(p);
    const int ng = p.G / ih;
    const int hq = item % ng;
    item /= ng;
    w.split = item % p.n_splits;
    item /= p.n_splits;
    w.hkv = item % p.Hkv;
    item /= p.Hkv;
    w.b = item % p.B;
    item /= p.B;
    const int qt = p.n_qtiles - 1 - item;  // longest causal tiles first
    w.h0 = w.hkv * p.G + hq * ih + (ih == 2 ? rank : 0);
    const int q0 = qt * rows;
    w.m0 = q0 + (rows == 256 ? rank * 128 : 0);
    const int qlast = min(q0 + rows, p.Lq) - 1;
    w.pmin = p.Lk - p.Lq + q0;
    w.pmax = p.Lk - p.Lq + qlast;
    lo = (p.causal && p.window) ? max(0, w.pmin - p.window + 1) : 0;
    hi = p.causal ? min(p.Lk, w.pmax + 1) : p.Lk;
    const int tlo = lo / BN, thi = (hi + BN - 1) / BN;
    const int per = (thi - tlo + p.n_splits - 1) / p.n_splits;
    w.t_begin = tlo + w.split * per;
    w.t_step = 1;
    w.t_count = max(0, min(per, thi - w.t_begin));
  } else {
    int hb;
    if (p.dec_cs > 0) {  // kDecode: the splits of one group are consecutive (one cluster each)
      w.split = item % p.n_splits;
      item /= p.n_splits;
      hb = item % p.n_hb;
      item /= p.n_hb;
    } else {
      hb = item % p.n_hb;
      item /= p.n_hb;
      w.split = item % p.n_splits;
      item /= p.n_splits;
    }
    w.hkv = item % p.Hkv;
    w.b = item / p.Hkv;
    w.h0 = w.hkv * p.G + hb * 16;
    w.m0 = 0;
    w.pmin = p.Lk - p.Lq;
    w.pmax = p.Lk - 1;
    lo = (p.causal && p.window) ? max(0, w.pmin - p.window + 1) : 0;
    hi = p.Lk;
    const int tlo = lo / BN, thi = (hi + BN - 1) / BN;
    const int S = p.n_splits;
    const int t0 = tlo + (((w.split - tlo) % S) + S) % S;
    w.t_begin = t0;
    w.t_step = S;
    w.t_count = t0 < thi ? (thi - 1 - t0) / S + 1 : 0;
  }
  return w;
}

// ------------------------------------------------------------ persistent schedule
// Items are the query tiles in make_work's order (longest causal tiles first,
// then batch, kv head and query head within its group).  With N items and U
// units, the first floor(N / U) * U items go out in whole waves, unit u taking
// item u of even waves and item U - 1 - u of odd ones (concurrent units work on
// neighbouring items, which share K/V rows in L2).  Of the r = N mod U leftover
// items, item i keeps its first min(T_i, L) key tiles on unit i; the remaining
// S_i = max(0, T_i - L) tiles of all of them are laid end to end and cut into
// equal contiguous shares for units r .. r + US - 1 (the host picks L, and
// passes US and the sum of S_i).  A suffix piece of item i on suffix unit k
// (counted from r) writes slot i + k, which is unique because i and k never both
// stay the same between two consecutive pieces.  Suffix units never wait, so
// the prefix units' waits end.

// Key tiles of a query tile (the same count make_work visits).
template <int BN, int QROWS>
__device__ __forceinline__ int item_tiles_for_qt(const AttnParams& p, int qt) {
  const int rows = tile_rows<QROWS>(p);
  const int q0 = qt * rows;
  const int qlast = min(q0 + rows, p.Lq) - 1;
  const int pmin = p.Lk - p.Lq + q0, pmax = p.Lk - p.Lq + qlast;
  const int lo = (p.causal && p.window) ? max(0, pmin - p.window + 1) : 0;
  const int hi = p.causal ? min(p.Lk, pmax + 1) : p.Lk;
  return (hi + BN - 1) / BN - lo / BN;
}

template <int BN, int QROWS>
__device__ __forceinline__ int item_tiles(const AttnParams& p, int idx) {
  return item_tiles_for_qt<BN, QROWS>(p, p.n_qtiles - 1 -
                                            idx / (p.G / item_heads<QROWS>(p) * p.Hkv * p.B));
}

// Work of item `idx`, key tiles [t0, t0 + cnt) of its visible range.
template <int BN, int QROWS>
__device__ __forceinline__ Work item_work(const AttnParams& p, int idx, int rank, int t0,
                                          int cnt) {
  Work w;
  int item = idx;
  const int ih = item_heads<QROWS>(p), rows = tile_rows<QROWS>(p);
  const int ng = p.G / ih;
  const int hq = item % ng;
  item /= ng;
  w.split = 0;
  w.hkv = item % p.Hkv;
  item /= p.Hkv;
  w.b = item % p.B;
  item /= p.B;
  const int qt = p.n_qtiles - 1 - item;
  w.h0 = w.hkv * p.G + hq * ih + (ih == 2 ? rank : 0);
  const int q0 = qt * rows;
  w.m0 = q0 + (rows == 256 ? rank * 128 : 0);
  const int qlast = min(q0 + rows, p.Lq) - 1;
  w.pmin = p.Lk - p.Lq + q0;
  w.pmax = p.Lk - p.Lq + qlast;
  const int lo = (p.causal && p.window) ? max(0, w.pmin - p.window + 1) : 0;
  w.t_begin = lo / BN + t0;
  w.t_step = 1;
  w.t_count = cnt;
  return w;
}

struct Piece {
  Work w;
  int kind;       // 0 whole item, 1 prefix (merges suffix slots), 2 suffix piece, 3 split partial
  int slot;       // kind 1: first suffix slot; kind 2: own slot
  int n_contrib;  // kind 1: suffix slots slot .. slot + n_contrib - 1, in key order
  int valid;      // 0 once the iterator is exhausted
};

// Position of one CTA in its sequence of pieces (plain data, so the softmax
// warps can keep it in shared memory).
struct IterState {
  long long pos, end;  // suffix unit: next suffix coordinate, end of its share
  long long A;         // suffix coordinate of leftover item i's first suffix tile
  long long L;         // prefix length of the leftover items
  long long SS;        // suffix tiles in all
  int stage;           // 0 waves, 1 leftover prefix, 2 suffix share, 3 done, 4 single piece
  int w, i;            // next wave; current leftover item
  int unit, rank;
  int n_full, r, US;
};

template <int BN, int QROWS>
__device__ __forceinline__ void iter_init(const AttnParams& p, IterState& st, int unit, int rank) {
  st.unit = unit;
  st.rank = rank;
  st.w = 0;
  st.i = 0;
  st.pos = st.end = st.A = 0;
  st.n_full = st.r = 0;
  st.L = p.tail_L;
  st.SS = p.tail_SS;
  st.US = p.tail_US;
  if (!p.persistent) {
    st.stage = 4;
    return;
  }
  const int N = p.n_qtiles * (p.G / item_heads<QROWS>(p)) * p.Hkv * p.B;
  const int U = p.n_units;
  st.n_full = N / U;
  st.r = N - st.n_full * U;
  st.stage = st.n_full > 0 ? 0 : 1;
  if (unit >= st.r) {
    const int k = unit - st.r;
    if (k < st.US) {
      st.pos = st.SS * k / st.US;
      st.end = st.SS * (k + 1) / st.US;
    }
  }
}

template <int BN, int QROWS>
__device__ __forceinline__ bool iter_next(const AttnParams& p, IterState& st, Piece& pc) {
  pc.valid = 0;
  pc.slot = 0;
  pc.n_contrib = 0;
  if (st.stage == 4) {  // one launch-planned piece per CTA
    st.stage = 3;
    pc.w = make_work<BN, QROWS>(p, st.unit, st.rank);
    pc.kind = p.write_partial ? 3 : 0;
    pc.valid = 1;
    return true;
  }
  const int U = p.n_units;
  if (st.stage == 0) {
    const int idx = st.w * U + ((st.w & 1) ? U - 1 - st.unit : st.unit);
    pc.w = item_work<BN, QROWS>(p, idx, st.rank, 0, item_tiles<BN, QROWS>(p, idx));
    pc.kind = 0;
    pc.valid = 1;
    if (++st.w == st.n_full) st.stage = 1;
    return true;
  }
  const int base = st.n_full * U;
  if (st.stage == 1) {
    if (st.unit < st.r) {
      // Prefix of leftover item `unit`; its suffix, if any, is on the suffix
      // units whose shares meet [A, A + S).
      st.stage = 3;
      const int i = st.unit;
      const int T = item_tiles<BN, QROWS>(p, base + i);
      const long long P = min(static_cast<long long>(T), st.L);
      const long long S = T - P;
      pc.w = item_work<BN, QROWS>(p, base + i, st.rank, 0, static_cast<int>(P));
      pc.kind = 0;
      if (S > 0) {
        long long A = 0;
        for (int j = 0; j < i; ++j) A += max(0ll, item_tiles<BN, QROWS>(p, base + j) - st.L);
        // suffix unit holding coordinate x: the largest k with SS * k / US <= x
        const long long kf = ((A + 1) * st.US - 1) / st.SS;
        const long long kl = ((A + S) * st.US - 1) / st.SS;
        pc.kind = 1;
        pc.slot = i + static_cast<int>(kf);
        pc.n_contrib = static_cast<int>(kl - kf + 1);
      }
      pc.valid = 1;
      return true;
    }
    st.stage = 2;
  }
  if (st.stage == 2) {
    if (st.pos >= st.end) {
      st.stage = 3;
      return false;
    }
    long long S = max(0ll, item_tiles<BN, QROWS>(p, base + st.i) - st.L);
    while (st.A + S <= st.pos) {
      st.A += S;
      ++st.i;
      S = max(0ll, item_tiles<BN, QROWS>(p, base + st.i) - st.L);
    }
    const long long stop = min(st.end, st.A + S);
    const int t0 = static_cast<int>(st.L + (st.pos - st.A));
    pc.w = item_work<BN, QROWS>(p, base + st.i, st.rank, t0, static_cast<int>(stop - st.pos));
    pc.kind = 2;
    pc.slot = st.i + (st.unit - st.r);
    pc.valid = 1;
    st.pos = stop;
    return true;
  }
  return false;
}

// Next piece of a CTA.  ONE (decode): a single launch-planned piece, without the
// persistent schedule's code.
template <int BN, int QROWS, bool ONE>
__device__ __forceinline__ bool next_piece(const AttnParams& p, IterState& st, Piece& pc) {
  if constexpr (ONE) {
    pc.valid = 0;
    pc.slot = 0;
    pc.n_contrib = 0;
    if (st.stage != 4) return false;
    st.stage = 3;
    pc.w = make_work<BN, QROWS>(p, st.unit, st.rank);
    pc.kind = 3;
    pc.valid = 1;
    return true;
  } else {
    return iter_next<BN, QROWS>(p, st, pc);
  }
}

// Bias entries for keys [k0, k0 + N) of one row, as N / 2 packed 16-bit pairs;
// keys at or past Lk (masked anyway) and rows without a bias (brow null) read 0.
template <int N>
__device__ __forceinline__ void load_bias(const uint16_t* brow, int k0, int Lk, bool vec,
                                          uint32_t (&bw)[N / 2]) {
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    const int kc = k0 + 8 * c;
    if (brow != nullptr && vec && kc + 8 <= Lk) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(brow + kc));
      bw[4 * c] = u.x;
      bw[4 * c + 1] = u.y;
      bw[4 * c + 2] = u.z;
      bw[4 * c + 3] = u.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t lo = (brow != nullptr && kc + e < Lk) ? __ldg(brow + kc + e) : 0u;
        const uint32_t hi = (brow != nullptr && kc + e + 1 < Lk) ? __ldg(brow + kc + e + 1) : 0u;
        bw[4 * c + e / 2] = lo | (hi << 16);
      }
    }
  }
}

// The two 16-bit values of a packed pair, widened (exactly) to float.
__device__ __forceinline__ float2 unpack2(uint32_t w, bool bf16) {
  if (bf16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// BIAS: add the caller's additive bias (p.bias) to the scores; the kernels
// without it never read p.bias.
template <bool BF16, int MODE, int HD, int HDV, bool BIAS = false>
__global__ void __launch_bounds__((Cfg<BF16, MODE, HD, HDV, BIAS>::NTHREADS), 1)
    attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<BF16, MODE, HD, HDV, BIAS>;
  constexpr bool PAIR = C::PAIR;
  constexpr bool DUO = C::DUO;
  constexpr bool CLUSTER = PAIR || DUO;
  constexpr int BN = C::BN;
  constexpr int HB = C::HB;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t sQ = sbase + C::Q_OFF;
  const uint32_t sRing = sbase + C::RING_OFF;
  const uint32_t sX = sbase + C::X_OFF;
  const uint32_t sBar = sbase + C::BAR_OFF;
  const uint32_t sP = sbase + C::P_OFF;  // P (Q in TMEM) / epilogue staging
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 244);
  float* red = reinterpret_cast<float*>(smem + C::RED_OFF);
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

  // The swizzled tiles need a 1024-byte aligned base; the dynamic shared window
  // provides it.  Should it ever not, fail cleanly instead of computing garbage.
  if ((sbase & 1023u) != 0) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevMisaligned);
    return;
  }
  // The 2-CTA variants address their peer's shared memory and pair their MMAs:
  // without a cluster of two that would touch memory that is not there.
  if ((CLUSTER && ptx::cluster_nctarank() != 2) ||
      (C::DEC && (p.dec_cs < 1 || ptx::cluster_nctarank() != static_cast<uint32_t>(p.dec_cs)))) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadCluster);
    return;
  }
  // Decode: every CTA is one split of one group.  A CTA beyond them (a grid
  // larger than planned) has nothing to compute and must not address memory;
  // its whole cluster is beyond them too, so no cluster barrier waits for it.
  if (C::DEC && static_cast<long long>(blockIdx.x) >=
                    static_cast<long long>(p.B) * p.Hkv * p.n_hb * p.n_splits) {
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadGrid);
    return;
  }
  // A merge kernel queued behind this grid may be placed on SMs as CTAs of this
  // grid finish (it waits for the whole grid before reading anything).
  ptx::griddep_launch_dependents();

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = CLUSTER ? ptx::cluster_ctarank() : 0u;
  const uint32_t peer = rank ^ 1u;
  // Item (one query tile, or one split of it) or, in persistent mode, unit index.
  // Persistent units are numbered from the end of the grid: blocks start in
  // index order, so should the grid not be resident all at once, the suffix
  // units (the highest unit numbers, which never wait) start first.
  const int cta_pair = CLUSTER ? static_cast<int>(blockIdx.x / 2) : static_cast<int>(blockIdx.x);
  const int item = p.persistent ? p.n_units - 1 - cta_pair : cta_pair;
  constexpr int QROWS = DUO ? 256 : 128;
  const int d0 = PAIR ? static_cast<int>(rank) * C::DH : 0;  // head-dim offset of this CTA
  // DUO: the pair's even CTA issues the MMAs and owns the barriers they wait on.
  auto leader_bar = [&](int i) -> uint32_t {
    return (DUO && rank != 0) ? ptx::mapa(bar(i), 0) : bar(i);
  };

  // Barriers are initialised by thread 0, or, in decode, by the producer lane,
  // which then starts its loads without waiting for the rest of the CTA.
  const bool init_thread =
      C::DEC ? (warp == C::kProducerWarp && lane == 0) : (threadIdx.x == 0);
  if (C::DEC && warp == C::kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&p.tm_k);
    ptx::prefetch_tmap(&p.tm_v);
  }
  if (init_thread) {
    ptx::mbar_init(bar(kBarQ), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      ptx::mbar_init(bar(kBarKvFull + s), 1);
      ptx::mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) ptx::mbar_init(bar(sfull_bar(b)), 1);
    ptx::mbar_init(bar(kBarPFull), C::kPFullArrivals);
    ptx::mbar_init(bar(kBarPvDone), 1);
    ptx::mbar_init(bar(kBarQFree), 1);
    ptx::mbar_init(bar(kBarOFree), C::kPFullArrivals);
    ptx::mbar_init(bar(kBarDrain), 1);
    if constexpr (C::PX) {
      for (int x = 0; x < C::X_SLOTS; ++x) {
        ptx::mbar_init(bar(xfull_bar(x)), 1);
        ptx::mbar_init(bar(xfree_bar(x)), 8);
        ptx::mbar_init(bar(xsready_bar<C::X_SLOTS>(x)), 4);
        ptx::mbar_init(bar(xsfree_bar<C::X_SLOTS>(x)), 8);
      }
      for (int b = 0; b < 2; ++b) ptx::mbar_init(bar(sfree_bar<C::X_SLOTS>(b)), 4);
    } else {
      ptx::mbar_init(bar(kBarXFull), 1);  // local expect_tx arrive + the peer's bulk-copy bytes
      ptx::mbar_init(bar(kBarXFree), 8);  // one arrive per softmax warp of the peer
      ptx::mbar_init(bar(kBarSFree), C::kPFullArrivals);
    }
    *abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  if (!C::DEC && warp == C::kProducerWarp && lane == 0) {
    if (!p.decode) ptx::prefetch_tmap(&p.tm_q);
    ptx::prefetch_tmap(&p.tm_k);
    ptx::prefetch_tmap(&p.tm_v);
  }
  // Decode: ring loads the producer issues right after initialising the
  // barriers, before the CTA-wide start (the first NSLOT slots need no wait:
  // each slot is used for the first time).  The producer loop skips them.
  uint32_t pre_issued = 0;
  if constexpr (C::DEC) {
    if (warp == C::kProducerWarp && lane == 0) {
      const Work w = make_work<C::BN, 128>(p, item, 0);
      const int bh_kv = w.b * p.Hkv + w.hkv;
      const int c = w.t_count;
      // Load units in the producer loop's order: K_0, then (K_j, V_{j-1}) for
      // j >= 1, then V_{c-1}.
      for (int u = 0; u < 2 * c && pre_issued < static_cast<uint32_t>(C::NSLOT); ++u) {
        const bool is_k = u == 0 || (u != 2 * c - 1 && (u & 1));
        const int j = u == 0 ? 0 : (u == 2 * c - 1 ? c - 1 : (is_k ? (u + 1) / 2 : u / 2 - 1));
        const int tile_key = (w.t_begin + j * w.t_step) * BN;
        const int key0 = p.kv_ring ? tile_key % p.kv_ring : tile_key;
        const int nsub = is_k ? C::KSUB : C::VSUB;
        for (int sub = 0; sub < nsub && pre_issued < static_cast<uint32_t>(C::NSLOT);
             ++sub, ++pre_issued) {
          const uint32_t slot = pre_issued;
          const uint32_t fb = bar(kBarKvFull + static_cast<int>(slot));
          ptx::mbar_arrive_expect_tx(fb, is_k ? C::K_SLOT_BYTES : C::V_SLOT_BYTES);
          if (is_k) {
            for (int e = 0; e < C::KBOX; ++e)
              ptx::tma_load_3d(sRing + slot * C::SLOT + e * (C::KROWS * 128), &p.tm_k, fb,
                               (sub * C::KBOX + e) * 64, key0, bh_kv);
          } else {
            for (int cc = 0; cc < C::VBOX; ++cc)
              ptx::tma_load_3d(sRing + slot * C::SLOT + cc * C::V_LBO, &p.tm_v, fb, cc * 64,
                               key0 + sub * C::VROWS, bh_kv);
          }
        }
      }
    }
  }
  if constexpr (C::DEC) {
    // Decode: each softmax thread copies its half of its row's query slice into
    // the swizzled query tile right away (16-byte chunk c of tile row t at
    // 16-byte position c ^ (t & 7) of the row's 128-byte line, one 16 KB block
    // per 64 columns); rows that hold no query row of this call are zeroed.
    if (warp < 8) {
      const Work w0 = make_work<C::BN, 128>(p, item, 0);
      const int t = (warp & 3) * 32 + lane;
      const int hl = t >> 3;
      const int i = ((((t & 7) - (p.Lk - p.Lq)) % 8) + 8) % 8;
      const int h = w0.h0 + hl;
      const bool valid = (i < p.Lq) && (hl < min(p.G, 16)) && (h < (w0.hkv + 1) * p.G);
      const long long rid = valid ? (static_cast<long long>(w0.b) * p.Hq + h) * p.Lq + i : 0;
      const uint16_t* src = p.q + rid * p.Dqk;
      const int hf = warp >> 2;
      for (int cq = hf * (C::DH / 16); cq < (hf + 1) * (C::DH / 16); ++cq) {
        const int dc = cq >> 3, cc = cq & 7;
        ptx::cp_async_16(sQ + dc * 16384 + t * 128 + ((cc ^ (t & 7)) << 4), src + cq * 8,
                         valid ? 16u : 0u);
      }
    }
  }
  if (warp == C::kMmaWarp) {
    if constexpr (DUO) {
      ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), 512);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
      ptx::tmem_relinquish();
    }
  }
  if constexpr (C::DEC) {
    // Named barriers instead of a CTA-wide one, so the producer never waits:
    // 6 (producer + MMA warps): the barriers are initialised;
    // 7 (MMA + softmax warps): tensor memory is allocated.
    if (warp == C::kProducerWarp) {
      __syncwarp();
      ptx::bar_arrive(6, 64);
    } else if (warp == C::kMmaWarp) {
      ptx::bar_sync(6, 64);
      ptx::tc_fence_before();
      ptx::bar_arrive(7, 288);
    } else if (warp < 8) {
      ptx::bar_sync(7, 288);
    }
  } else {
    ptx::tc_fence_before();
    __syncthreads();
    if (CLUSTER) ptx::cluster_sync();  // peer barriers initialised before any remote use
  }
  ptx::tc_fence_after();
  // (in decode the producer and idle warps never use it and do not wait for it)
  const uint32_t tmem = (C::DEC && warp >= 8 && warp != C::kMmaWarp) ? 0u : *tmem_slot;
  const bool mma_cta = !DUO || rank == 0;  // this CTA issues MMAs

  // Producer / MMA bookkeeping kept for the drain after an abort.
  int issued_q = 0;  // query tiles loaded (one per piece with key tiles)
  uint32_t ring_issued = pre_issued;  // ring loads issued, in sequence order
  int mma_issued = 0;

  // Warpgroup 2 (producer, MMA issuer, two idle warps) hands its spare
  // registers to the softmax warpgroups; each side changes its budget inside its
  // own branch, so the code after a change is that side's alone.
  if (warp >= C::kProducerWarp) {
  ptx::setmaxnreg_dec<C::kRegsOther>();
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      auto load = [&](uint32_t dst, const CUtensorMap* m, uint32_t fullbar, int c0, int c1,
                      int c2) {
        if constexpr (DUO)
          ptx::tma_load_3d_pair(dst, m, fullbar, c0, c1, c2);
        else
          ptx::tma_load_3d(dst, m, fullbar, c0, c1, c2);
      };
      uint32_t n = 0;  // ring sequence number, continued across pieces
      bool ok = true;
      // Iterator in shared memory: it stays out of this warpgroup's small
      // register budget.
      IterState& ist = *reinterpret_cast<IterState*>(smem + C::ITER_OFF + 256);
      Piece& pc = *reinterpret_cast<Piece*>(smem + C::ITER_OFF + 256 + 96);
      iter_init<BN, QROWS>(p, ist, item, static_cast<int>(rank));
      while (ok && next_piece<BN, QROWS, C::DEC>(p, ist, pc)) {
        const Work& w = pc.w;
        const int count = w.t_count;
        if (count == 0) continue;
        const int bh_q = w.b * p.Hq + w.h0;
        const int bh_kv = w.b * p.Hkv + w.hkv;
        if (!p.decode && p.withhold_q != 1) {
          // The query buffer is free once the previous piece's last S has completed.
          if (issued_q > 0 && !wait_bar(bar(kBarQFree), (issued_q - 1) & 1, abort_flag, p.status,
                                        kDevTimeoutQ)) {
            ok = false;
            break;
          }
          const uint32_t qbar = leader_bar(kBarQ);
          if (mma_cta) ptx::mbar_arrive_expect_tx(bar(kBarQ), DUO ? 2 * C::Q_BYTES : C::Q_BYTES);
          for (int c = 0; c < C::DH / 64; ++c)
            load(sQ + c * 16384, &p.tm_q, qbar, d0 + c * 64, w.m0, bh_q);
          ++issued_q;
        }
        // Row of the first key of a tile (tiles never straddle a ring's end: the
        // ring length is a multiple of 128 and tiles start at multiples of BN).
        auto kv_row = [&](int key) -> int { return p.kv_ring ? key % p.kv_ring : key; };
        auto next_slot = [&](int& slot, uint32_t& fullbar, uint32_t bytes) -> bool {
          slot = n % C::NSLOT;
          if (!wait_bar(bar(kBarKvEmpty + slot), ((n / C::NSLOT) & 1) ^ 1, abort_flag, p.status,
                        kDevTimeoutKvEmpty))
            return false;
          fullbar = leader_bar(kBarKvFull + slot);
          // The MMA CTA posts the bytes of both halves (DUO) on its own barrier.
          if (mma_cta)
            ptx::mbar_arrive_expect_tx(bar(kBarKvFull + slot), DUO ? 2 * bytes : bytes);
          return true;
        };
        auto load_k = [&](int j) {
          // DUO: CTA `rank` loads keys [64 rank, 64 rank + 64) of the 128-key tile.
          const int key0 =
              kv_row((w.t_begin + j * w.t_step) * BN) + (DUO ? static_cast<int>(rank) * 64 : 0);
          for (int ks = 0; ks < C::KSUB && ok; ++ks, ++n) {
            if (n < pre_issued) continue;  // issued before the CTA-wide start
            int slot;
            uint32_t fb;
            if (!next_slot(slot, fb, C::K_SLOT_BYTES)) {
              ok = false;
              break;
            }
            for (int e = 0; e < C::KBOX; ++e)
              load(sRing + slot * C::SLOT + e * (C::KROWS * 128), &p.tm_k, fb,
                   d0 + (ks * C::KBOX + e) * 64, key0, bh_kv);
            ring_issued = n + 1;
          }
        };
        auto load_v = [&](int j) {
          // DUO: CTA `rank` loads head-dim columns [DH/2 rank, DH/2 (rank + 1)) of V.
          const int key0 = kv_row((w.t_begin + j * w.t_step) * BN);
          const int dv0 = DUO ? static_cast<int>(rank) * (C::DV / 2) : d0;
          for (int vs = 0; vs < C::VSUB && ok; ++vs, ++n) {
            if (n < pre_issued) continue;  // issued before the CTA-wide start
            int slot;
            uint32_t fb;
            if (!next_slot(slot, fb, C::V_SLOT_BYTES)) {
              ok = false;
              break;
            }
            for (int c = 0; c < C::VBOX; ++c)
              load(sRing + slot * C::SLOT + c * C::V_LBO, &p.tm_v, fb, dv0 + c * 64,
                   key0 + vs * C::VROWS, bh_kv);
            ring_issued = n + 1;
          }
        };
        // The MMA issuer consumes the ring in this order: K of tile j comes
        // S_AHEAD tiles before V of tile j - S_AHEAD.
        for (int j = 0; j < count + C::S_AHEAD && ok; ++j) {
          if (j < count) load_k(j);
          if (ok && j >= C::S_AHEAD) load_v(j - C::S_AHEAD);
        }
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && mma_cta) {
      bool ok = true;
      uint32_t n = 0;   // ring sequence number, continued across pieces
      int g0 = 0;       // global index of the piece's first key tile (barrier phases)
      int done_pieces = 0;
      auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
        if constexpr (DUO)
          ptx::mma_f16_ss_pair(d, a, b, idesc, acc);
        else
          ptx::mma_f16_ss(d, a, b, idesc, acc);
      };
      auto commit = [&](int barid) {  // to this barrier in every CTA that waits on it
        if constexpr (DUO)
          ptx::mma_commit_pair_mc(bar(barid), 3);
        else
          ptx::mma_commit(bar(barid));
      };
      auto consume = [&](uint32_t& slot_addr) -> bool {
        const int slot = n % C::NSLOT;
        if (!wait_bar(bar(kBarKvFull + slot), (n / C::NSLOT) & 1, abort_flag, p.status,
                      kDevTimeoutKvFull))
          return false;
        ptx::tc_fence_after();
        slot_addr = sRing + slot * C::SLOT;
        return true;
      };
      auto release = [&]() {
        commit(kBarKvEmpty + static_cast<int>(n % C::NSLOT));
        ++n;
      };
      auto do_s = [&](int gt) {
        // Q in TMEM: the single S buffer is free once the softmax has read
        // S_{gt-1}.  Otherwise S buffer gt % 2 last held S_{gt-2} and then
        // P_{gt-2}; the P.V of tile gt - 2 that reads P was issued before this
        // product, and the tensor pipe runs one thread's MMAs in issue order.
        if constexpr (C::SFREE) {
          // The S buffer is free once its scores have been read (kDuoQ: by
          // every softmax warp; kPairX: by the exchange warps).
          if (gt >= C::NSBUF) {
            const uint32_t gu = static_cast<uint32_t>(gt);
            if (!wait_bar<DUO>(bar(sfree_bar<C::X_SLOTS>(static_cast<int>(gu % C::NSBUF))),
                               (gu / C::NSBUF - 1) & 1, abort_flag, p.status, kDevTimeoutSEmpty)) {
              ok = false;
              return;
            }
            ptx::tc_fence_after();
          }
        }
        const uint32_t d_tmem = tmem + C::S_COL + (static_cast<uint32_t>(gt) % C::NSBUF) * BN;
        for (int ks = 0; ks < C::KSUB; ++ks) {
          uint32_t sk;
          if (!consume(sk)) {
            ok = false;
            return;
          }
#pragma unroll
          for (int e = 0; e < C::KBOX; ++e) {
            const int dc = ks * C::KBOX + e;  // 64-column chunk of the head dim
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t b =
                  ptx::sdesc_sw128(sk + e * (C::KROWS * 128) + kk * 32, 16, 1024);
              if constexpr (C::QTM) {
                // A = Q from tensor memory: head-dim columns [16 (4 dc + kk), +16)
                // at TMEM columns Q_COL + 8 (4 dc + kk).
                const uint32_t a = tmem + C::Q_COL + static_cast<uint32_t>((dc * 4 + kk) * 8);
                if constexpr (DUO)
                  ptx::mma_f16_ts_pair(d_tmem, a, b, C::IDESC_QK, (dc | kk) != 0);
                else
                  ptx::mma_f16_ts(d_tmem, a, b, C::IDESC_QK, (dc | kk) != 0);
              } else {
                const uint64_t a = ptx::sdesc_sw128(sQ + dc * 16384 + kk * 32, 16, 1024);
                mma(d_tmem, a, b, C::IDESC_QK, (dc | kk) != 0);
              }
            }
          }
          release();
          ++mma_issued;
        }
        commit(sfull_bar(static_cast<int>(static_cast<uint32_t>(gt) % C::NSBUF)));
      };
      auto do_pv = [&](int gt, int j) {  // j: tile index within the piece
        if (!wait_bar<DUO>(bar(kBarPFull), gt & 1, abort_flag, p.status, kDevTimeoutPFull)) {
          ok = false;
          return;
        }
        if (j == 0 && done_pieces > 0) {
          // The first product of a piece overwrites O: the previous piece's
          // epilogue must have read it.
          if (!wait_bar<DUO>(bar(kBarOFree), (done_pieces - 1) & 1, abort_flag, p.status,
                             kDevTimeoutPvDone)) {
            ok = false;
            return;
          }
        }
        ptx::tc_fence_after();
        for (int vs = 0; vs < C::VSUB; ++vs) {
          uint32_t sv;
          if (!consume(sv)) {
            ok = false;
            return;
          }
#pragma unroll
          for (int kk = 0; kk < C::VROWS / 16; ++kk) {
            const int key = vs * C::VROWS + kk * 16;
            const uint64_t b = ptx::sdesc_sw128(sv + kk * 2048, C::V_LBO, 1024);
            if constexpr (C::PSM) {
              // A = P_gt in shared memory (K-major, 128B-swizzled, 64 keys a row).
              const uint64_t a =
                  ptx::sdesc_sw128(sP + (key / 64) * 16384 + (key % 64) * 2, 16, 1024);
              mma(tmem, a, b, C::IDESC_PV, (j | vs | kk) != 0);
            } else {
              // A = P_gt in tensor memory (keys key..key+15 at columns key / 2).
              const uint32_t a =
                  tmem + C::S_COL + (static_cast<uint32_t>(gt) % C::NSBUF) * BN + key / 2;
              if constexpr (DUO)
                ptx::mma_f16_ts_pair(tmem, a, b, C::IDESC_PV, (j | vs | kk) != 0);
              else
                ptx::mma_f16_ts(tmem, a, b, C::IDESC_PV, (j | vs | kk) != 0);
            }
          }
          release();
          ++mma_issued;
        }
        commit(kBarPvDone);
      };
      IterState& ist = *reinterpret_cast<IterState*>(smem + C::ITER_OFF + 512);
      Piece& pc = *reinterpret_cast<Piece*>(smem + C::ITER_OFF + 512 + 96);
      iter_init<BN, QROWS>(p, ist, item, static_cast<int>(rank));
      while (ok && next_piece<BN, QROWS, C::DEC>(p, ist, pc)) {
        const int count = pc.w.t_count;
        if (count == 0) continue;
        if (!wait_bar(bar(kBarQ), done_pieces & 1, abort_flag, p.status, kDevTimeoutQ)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if constexpr (C::QTM) {
          // Q to tensor memory, 16 head-dim columns per copy; the previous
          // piece's last Q.K^T, issued before, has read the old Q.  The query
          // buffer in shared memory is free once these copies have completed.
          for (int dc = 0; dc < C::DH / 64; ++dc)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t dst = tmem + C::Q_COL + static_cast<uint32_t>((dc * 4 + kk) * 8);
              const uint64_t src = ptx::sdesc_sw128(sQ + dc * 16384 + kk * 32, 16, 1024);
              if constexpr (DUO)
                ptx::tmem_cp_128x256b_pair(dst, src);
              else
                ptx::tmem_cp_128x256b(dst, src);
            }
          commit(kBarQFree);
        }
        // S_j is issued S_AHEAD products ahead of P_{j-S_AHEAD}.V; its buffer last
        // held S / P of tile j - NSBUF, whose P.V was issued before it (one
        // thread's MMAs run in issue order).
        if constexpr (C::S_AHEAD == 1) {
          do_s(g0);
          if (!C::QTM && ok && count == 1) commit(kBarQFree);
          for (int j = 1; j < count && ok; ++j) {
            do_s(g0 + j);
            if (!C::QTM && ok && j == count - 1) commit(kBarQFree);
            if (ok) do_pv(g0 + j - 1, j - 1);
          }
          if (ok) do_pv(g0 + count - 1, count - 1);
        } else {
          const int pro = min(count, C::S_AHEAD);
          for (int j = 0; j < pro && ok; ++j) {
            do_s(g0 + j);
            if (!C::QTM && ok && j == count - 1) commit(kBarQFree);
          }
          for (int j = C::S_AHEAD; j < count && ok; ++j) {
            do_s(g0 + j);
            if (!C::QTM && ok && j == count - 1) commit(kBarQFree);
            if (ok) do_pv(g0 + j - C::S_AHEAD, j - C::S_AHEAD);
          }
          for (int j = count - pro; j < count && ok; ++j) do_pv(g0 + j, j);
        }
        g0 += count;
        ++done_pieces;
      }
    }
  }
  if constexpr (C::DEC) {
    // The softmax warps' cluster merge: this warpgroup takes part in its
    // cluster barriers (every thread of the cluster arrives at each; the
    // second one is waited for at teardown).
    __syncwarp();
    ptx::cluster_sync();
    ptx::cluster_arrive();
  }
  } else if (C::PX && warp >= C::kExchangeWarp) {
    ptx::setmaxnreg_dec<C::kRegsExchange>();
    // ------------------------------------------------------------ exchange (kPairX)
    // One thread per row (warp 8 + q reads TMEM lanes [32q, 32q + 32)).  Per
    // key tile j (S buffer j mod 2, exchange slot j mod X_SLOTS): read this
    // CTA's partial scores from TMEM (then the MMA may reuse the buffer), stage
    // them in XS once our softmax warps and the peer's have read the slot's
    // previous tile, and bulk-copy each warp's block into the peer's X slot.
    // One thread posts the bytes the peer sends into our X slot.  The softmax
    // warps add the halves.  (kPairXD keeps one exchange slot, so that its
    // shared memory holds an 8-slot ring; kPairX keeps two.)
    const int q4 = warp & 3;
    const int t = q4 * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const Work w = make_work<BN, QROWS>(p, item, static_cast<int>(rank));
    const int count = w.t_count;
    bool row_valid = true;
    if (p.decode) {
      const int hl = t >> 3;
      const int i = ((((t & 7) - (p.Lk - p.Lq)) % 8) + 8) % 8;
      row_valid = (i < p.Lq) && (hl < min(p.G, 16)) && (w.h0 + hl < (w.hkv + 1) * p.G);
    }
    // Rows whose partial scores go through the exchange: every row in prefill,
    // the real query rows in decode, packed in row order within each warp.  A
    // row's BN scores (256 bytes) sit at 16-byte chunk g ^ (position mod 16).
    const uint32_t xmask = p.decode ? __ballot_sync(0xffffffffu, row_valid) : 0xffffffffu;
    const uint32_t xidx = __popc(xmask & ((1u << lane) - 1u));
    const bool xrow = (xmask >> lane) & 1u;
    const uint32_t nrows = __popc(xmask);
    constexpr uint32_t RB = BN * 4;
    const uint32_t wofs = static_cast<uint32_t>(q4) * (32 * RB);
    const uint32_t rofs = wofs + xidx * RB;
    const uint32_t xsw = xidx & 15u;
    uint32_t xbytes = C::X_BYTES;  // bytes the peer sends per tile
    if (p.decode) {
      int nv = 0;
      for (int r = 0; r < 128; ++r) {
        const int ri = ((((r & 7) - (p.Lk - p.Lq)) % 8) + 8) % 8;
        nv += (ri < p.Lq) && ((r >> 3) < min(p.G, 16)) && (w.h0 + (r >> 3) < (w.hkv + 1) * p.G);
      }
      xbytes = static_cast<uint32_t>(nv) * RB;
    }
    auto arrive_local = [&](int barid) {  // one arrival per warp
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(barid));
    };
    bool alive = true;
    for (int j = 0; j < count && alive; ++j) {
      const int b = j & 1;  // S buffer
      const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
      const int xb = j % C::X_SLOTS;  // X / XS slot
      const uint32_t xph = static_cast<uint32_t>(j / C::X_SLOTS) & 1u;
      alive = __all_sync(0xffffffffu, wait_bar(bar(sfull_bar(b)), ph, abort_flag, p.status,
                                               kDevTimeoutSFull));
      if (!alive) break;
      ptx::tc_fence_after();
      uint32_t r0[32], r1[32];
      ptx::tmem_ld32(lane_base + C::S_COL + b * BN, r0);
      ptx::tmem_ld32(lane_base + C::S_COL + b * BN + 32, r1);
      ptx::tmem_wait_ld();
      ptx::reg_fence(r0);
      ptx::reg_fence(r1);
      ptx::tc_fence_before();
      arrive_local(sfree_bar<C::X_SLOTS>(b));
      alive = __all_sync(0xffffffffu, wait_bar(bar(xsfree_bar<C::X_SLOTS>(xb)), xph ^ 1u,
                                               abort_flag, p.status, kDevTimeoutXFree));
      if (alive)
        alive = __all_sync(0xffffffffu, wait_bar<true>(bar(xfree_bar(xb)), xph ^ 1u, abort_flag,
                                                       p.status, kDevTimeoutXFree));
      if (!alive) break;
      const uint32_t xs = sbase + C::XS_OFF + static_cast<uint32_t>(xb) * C::X_BYTES;
      if (xrow) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           xs + rofs + ((static_cast<uint32_t>(g) ^ xsw) << 4)),
                       "r"(r0[4 * g]), "r"(r0[4 * g + 1]), "r"(r0[4 * g + 2]), "r"(r0[4 * g + 3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           xs + rofs + ((static_cast<uint32_t>(g + 8) ^ xsw) << 4)),
                       "r"(r1[4 * g]), "r"(r1[4 * g + 1]), "r"(r1[4 * g + 2]), "r"(r1[4 * g + 3])
                       : "memory");
        }
      }
      ptx::fence_proxy_async_smem();
      arrive_local(xsready_bar<C::X_SLOTS>(xb));  // our softmax warps may read the slot
      if (threadIdx.x == C::kExchangeWarp * 32)
        ptx::mbar_arrive_expect_tx(bar(xfull_bar(xb)), xbytes);
      if (lane == 0 && nrows > 0)
        ptx::bulk_copy_to_peer(ptx::mapa(sX + static_cast<uint32_t>(xb) * C::X_BYTES + wofs, peer),
                               xs + wofs, nrows * RB, ptx::mapa(bar(xfull_bar(xb)), peer));
    }
  } else {
    ptx::setmaxnreg_inc<C::kRegsSoftmax>();
    // ------------------------------------------------------------ softmax / epilogue
    // Two threads per row: warps q and q+4 read TMEM lanes [32q, 32q+32); `half`
    // selects which half of the key columns (and of the O columns) a thread owns.
    const int q4 = warp & 3;
    const int half = warp >> 2;
    const int t = q4 * 32 + lane;  // row of the tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    // Per-warp arrival on a barrier the MMA issuer waits on.  In the odd CTA of
    // a 2-SM pair the barrier is the even CTA's: for P-ready, the P rows stay in
    // this CTA and are read by this SM's tensor core (the fence.proxy.async
    // before the arrive makes them visible to it); for O-free, this CTA's reads
    // of its own tensor memory have completed.  A CTA-scope release suffices.
    auto warp_arrive = [&](int barid) {
      __syncwarp();
      if (lane == 0) {
        if (DUO && rank != 0)
          ptx::mbar_arrive_remote_cta(ptx::mapa(bar(barid), 0));
        else
          ptx::mbar_arrive(bar(barid));
      }
    };

    const float c = p.c;
    const float cs = BIAS ? 1.f : c;  // factor from the scores held in s to log2 units
    constexpr float kLog2e = 1.4426950408889634f;
    bool ok = true;      // false once the two halves of this row pair agree to stop
    bool alive = true;   // false once a wait of this warp gave up
    int use = 0;  // pair-barrier uses so far
    const uint32_t pair_id = 2 + q4;  // named barrier of warps q4 and q4 + 4
    int g0 = 0;   // global index of the piece's first key tile (barrier phases)

    // Swap one float per row with the other half of the row.  The named barrier
    // also ANDs `alive` across the 64 threads, so both warps of a pair always
    // take the same decision to stop and neither is left waiting at a barrier.
    auto swap_half = [&](float mine, float& other) -> bool {
      float* slot = red + (use & 1) * 256;
      slot[half * 128 + t] = mine;
      const bool both = ptx::bar_red_and(pair_id, 64, alive);
      other = slot[(half ^ 1) * 128 + t];
      ++use;
      return both;
    };

    // The piece iterator lives in shared memory: thread 0 advances it, and every
    // piece starts at a named barrier over all 256 softmax threads that also
    // ANDs their `ok`, so all of them agree whether to go on.
    IterState* ist = reinterpret_cast<IterState*>(smem + C::ITER_OFF);
    static_assert(sizeof(IterState) <= 96 && 96 + 2 * sizeof(Piece) <= 256,
                  "iterator area holds the state and two pieces");
    Piece* pcs = reinterpret_cast<Piece*>(smem + C::ITER_OFF + 96);  // two, by piece parity
    const int unit = item;
    if (threadIdx.x == 0) iter_init<BN, QROWS>(p, *ist, unit, static_cast<int>(rank));
    for (int np = 0;; ++np) {
      if (threadIdx.x == 0) next_piece<BN, QROWS, C::DEC>(p, *ist, pcs[np & 1]);
      if (!ptx::bar_red_and(1, 256, ok)) break;
      const Piece& pc = pcs[np & 1];
      if (!pc.valid) break;
      const Work& w = pc.w;
      const int count = w.t_count;
      int row_p;            // bottom-right position of this row
      bool row_valid;
      long long row_id;     // flat (b, h, i) row index, -1 if none
      const uint16_t* brow = nullptr;  // this row's bias entries (key 0), if any
      if (!p.decode) {
        const int i = w.m0 + t;
        row_valid = i < p.Lq;
        row_p = p.Lk - p.Lq + min(i, p.Lq - 1);
        row_id = row_valid ? (static_cast<long long>(w.b) * p.Hq + w.h0) * p.Lq + i : -1;
        if (BIAS && row_valid)
          brow = p.bias + w.b * p.bias_sb + w.h0 * p.bias_sh + i * p.bias_sq;
      } else {
        const int hl = t >> 3;
        const int slot = t & 7;
        const int base = p.Lk - p.Lq;
        const int i = (((slot - base) % 8) + 8) % 8;
        const int h = w.h0 + hl;
        row_valid = (i < p.Lq) && (hl < min(p.G, 16)) && (h < (w.hkv + 1) * p.G);
        row_p = base + (row_valid ? i : 0);
        row_id = row_valid ? (static_cast<long long>(w.b) * p.Hq + h) * p.Lq + i : -1;
        if (BIAS && row_valid)
          brow = p.bias + w.b * p.bias_sb + h * p.bias_sh + i * p.bias_sq;
        if (count > 0) {
          // Decode: stage this thread's half of the row's query slice into the
          // swizzled Q tile (16-byte chunks of 8 elements); kDecode issued
          // these copies at entry and only waits for them here, kPairXD
          // issues all of a thread's loads before its first store.
          if constexpr (C::DEC) {
            ptx::cp_async_wait_all();
          } else if constexpr (C::PXD) {
            const uint4* src =
                reinterpret_cast<const uint4*>(p.q + row_id * p.Dqk + d0) + half * (C::DH / 16);
            uint4 v[C::DH / 16];
#pragma unroll
            for (int c = 0; c < C::DH / 16; ++c)
              v[c] = row_valid ? src[c] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < C::DH / 16; ++c) {
              const int cq = half * (C::DH / 16) + c;
              const int dc = cq >> 3, cc = cq & 7;
              const uint32_t addr = sQ + dc * 16384 + t * 128 + ((cc ^ (t & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[c].x),
                           "r"(v[c].y), "r"(v[c].z), "r"(v[c].w)
                           : "memory");
            }
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + row_id * p.Dqk + d0);
            for (int cq = half * (C::DH / 16); cq < (half + 1) * (C::DH / 16); ++cq) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (row_valid) v = src[cq];
              const int dc = cq >> 3, cc = cq & 7;
              const uint32_t addr = sQ + dc * 16384 + t * 128 + ((cc ^ (t & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x),
                           "r"(v.y), "r"(v.z), "r"(v.w)
                           : "memory");
            }
          }
          ptx::fence_proxy_async_smem();
          asm volatile("bar.sync 1, 256;" ::: "memory");
          if (threadIdx.x == 0 && p.withhold_q != 1) ptx::mbar_arrive(bar(kBarQ));
        }
      }

      // Pair: rows of this warp whose partial scores go through the exchange
      // (the exchange warps pack them the same way): every row in prefill, the
      // real query rows in decode (16 x Lq of the 128), in row order.
      const uint32_t xmask =
          (PAIR && p.decode) ? __ballot_sync(0xffffffffu, row_valid) : 0xffffffffu;
      const uint32_t xidx = __popc(xmask & ((1u << lane) - 1u));  // packed position
      const bool xrow = (xmask >> lane) & 1u;

      float m_run = -INFINITY;  // running max of c * s (lazy: the true max may exceed it by < 8)
      float l = 0.f;            // this half's share of the row sum

      for (int j = 0; j < count; ++j) {
        const int gt = g0 + j;
        const int tile = w.t_begin + j * w.t_step;
        const int kb = tile * BN + half * HB;  // first key of this thread's columns
        const int buf = static_cast<int>(static_cast<uint32_t>(gt) % C::NSBUF);  // S buffer
        float s[HB];
#pragma unroll
        for (int e = 0; e < HB; ++e) s[e] = -INFINITY;
        // Bias: this tile's entries are requested before the wait for S, and the
        // next tile's lines are prefetched into L2.
        uint32_t bw[BIAS ? HB / 2 : 1];
        if constexpr (BIAS) {
          load_bias<HB>(brow, kb, p.Lk, p.bias_vec != 0, bw);
          if (brow != nullptr && j + 1 < count) {
            const int kn = (tile + w.t_step) * BN + half * HB;
            if (kn < p.Lk) ptx::prefetch_l2(brow + kn);
            if (kn + HB - 1 < p.Lk) ptx::prefetch_l2(brow + kn + HB - 1);
          }
        }
        if constexpr (C::PX) {
          // The exchange warps have staged this CTA's partial scores of tile j
          // in XS slot j mod X_SLOTS and the peer's have landed in that X slot:
          // add this thread's half of the row (chunks half * 8 .. of the row's
          // 16, at chunk g ^ (row position mod 16)), then hand both slots back.
          const int bx = gt % C::X_SLOTS;
          const uint32_t phx = static_cast<uint32_t>(gt / C::X_SLOTS) & 1u;
          if (alive)
            alive = __all_sync(0xffffffffu, wait_bar(bar(xsready_bar<C::X_SLOTS>(bx)), phx, abort_flag,
                                                     p.status, kDevTimeoutXFull));
          if (alive)
            alive = __all_sync(0xffffffffu, wait_bar<true>(bar(xfull_bar(bx)), phx, abort_flag,
                                                           p.status, kDevTimeoutXFull));
          if (alive && xrow) {
            const uint32_t rb = static_cast<uint32_t>(q4) * (32 * BN * 4) + xidx * (BN * 4);
            const uint32_t xs = sbase + C::XS_OFF + static_cast<uint32_t>(bx) * C::X_BYTES + rb;
            const uint32_t xr = sX + static_cast<uint32_t>(bx) * C::X_BYTES + rb;
            const uint32_t sw = xidx & 15u;
#pragma unroll
            for (int g = 0; g < HB / 4; ++g) {
              const uint32_t off = (static_cast<uint32_t>(half * (HB / 4) + g) ^ sw) << 4;
              float a0, a1, a2, a3, b0, b1, b2, b3;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3)
                           : "r"(xs + off)
                           : "memory");
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3)
                           : "r"(xr + off)
                           : "memory");
              // rank 0 adds (own + peer), rank 1 adds (peer + own): the same
              // two operands, so both CTAs hold bit-identical scores.
              s[4 * g] = a0 + b0;
              s[4 * g + 1] = a1 + b1;
              s[4 * g + 2] = a2 + b2;
              s[4 * g + 3] = a3 + b3;
            }
          }
          if (alive) {
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(bar(xsfree_bar<C::X_SLOTS>(bx)));
              ptx::mbar_arrive_remote_cta(ptx::mapa(bar(xfree_bar(bx)), peer));
            }
          }
        } else {
          if (alive)
            alive = __all_sync(0xffffffffu,
                               wait_bar(bar(sfull_bar(buf)), (static_cast<uint32_t>(gt) / C::NSBUF) & 1,
                                        abort_flag, p.status, kDevTimeoutSFull));
          if (BIAS && alive) {
            // Scores straight to the log2 domain, c * s + log2(e) * bias, one
            // 32-column chunk at a time (a masked key becomes -inf below).
            ptx::tc_fence_after();
#pragma unroll
            for (int cch = 0; cch < HB / 32; ++cch) {
              uint32_t r[32];
              ptx::tmem_ld32(lane_base + C::S_COL + buf * BN + half * HB + cch * 32, r);
              ptx::tmem_wait_ld();
              ptx::reg_fence(r);
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float2 bv = unpack2(bw[(cch * 32 + e) / 2], BF16);
                s[cch * 32 + e] = fmaf(__uint_as_float(r[e]), c, bv.x * kLog2e);
                s[cch * 32 + e + 1] = fmaf(__uint_as_float(r[e + 1]), c, bv.y * kLog2e);
              }
            }
          } else if (alive) {
            ptx::tc_fence_after();
            uint32_t r[HB / 32][32];
#pragma unroll
            for (int cch = 0; cch < HB / 32; ++cch)
              ptx::tmem_ld32(lane_base + C::S_COL + buf * BN + half * HB + cch * 32, r[cch]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int cch = 0; cch < HB / 32; ++cch) {
              ptx::reg_fence(r[cch]);
#pragma unroll
              for (int e = 0; e < 32; ++e) s[cch * 32 + e] = __uint_as_float(r[cch][e]);
            }
          }
          if constexpr (C::QTM) {
            // Single S buffer: the next Q.K^T may overwrite it once every softmax
            // warp has read its lanes (the loads above have completed).
            if (alive) {
              ptx::tc_fence_before();
              warp_arrive(kBarSFree);
            }
          }
        }

        // Mask (only on tiles that straddle the band edge or the end of the keys).
        const int tb = tile * BN;
        const bool edge = (tb + BN > p.Lk) || (p.causal && tb + BN - 1 > w.pmin) ||
                          (p.causal && p.window && tb < w.pmax - p.window + 1);
        if (edge) {
          if constexpr (PAIR) {
            // (The pairs keep the per-key test: the range form below measured
            // 20% slower in their prefill, through code generation alone.)
#pragma unroll
            for (int e = 0; e < HB; ++e) {
              const int kj = kb + e;
              const bool vis = kj < p.Lk && (!p.causal || kj <= row_p) &&
                               (!p.window || row_p - kj < p.window);
              s[e] = vis ? s[e] : -INFINITY;
            }
          } else {
            // Key kb + e is visible iff lo <= e <= hi: below Lk, at or before
            // the row's position (causal), and within the window (a window
            // implies causal).
            int hi = p.Lk - 1;
            if (p.causal) hi = min(hi, row_p);
            const int lo = p.window ? row_p - p.window + 1 - kb : -kb;
            hi -= kb;
#pragma unroll
            for (int e = 0; e < HB; ++e) s[e] = (e >= lo && e <= hi) ? s[e] : -INFINITY;
          }
        }
        // Pair with a bias: the summed scores move to the log2 domain here (-inf,
        // from the mask or the bias, stays -inf).  With a bias cs = 1 below.
        if constexpr (BIAS && PAIR) {
#pragma unroll
          for (int e = 0; e < HB; e += 2) {
            const float2 bv = unpack2(bw[e / 2], BF16);
            s[e] = fmaf(s[e], c, bv.x * kLog2e);
            s[e + 1] = fmaf(s[e + 1], c, bv.y * kLog2e);
          }
        }
        // Row max: tree over this half, then swap with the other half.
        float mh;
        {
          float mm[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mm[k] = s[k];
#pragma unroll
          for (int e = 8; e < HB; ++e) mm[e & 7] = fmaxf(mm[e & 7], s[e]);
          mh = fmaxf(fmaxf(fmaxf(mm[0], mm[1]), fmaxf(mm[2], mm[3])),
                     fmaxf(fmaxf(mm[4], mm[5]), fmaxf(mm[6], mm[7])));
        }
        float mo;
        ok = swap_half(mh, mo);
        if (!ok) break;  // both halves of the row stop together
        const float xm = fmaxf(mh, mo) * cs;  // cs > 0, so -inf stays -inf
        const bool grow = xm > m_run + 8.0f;
        const float m_old = m_run;
        const bool rescale_o = grow && (m_old != -INFINITY) && (j > 0);
        float alpha = 1.f;
        if (grow) {
          alpha = ptx::ex2(m_old - xm);  // 0 when m_old == -inf
          l *= alpha;
          m_run = xm;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;

        // Probabilities 2^(cs*s - m), partial row sum, pack to 16-bit pairs.
        uint32_t pk[HB / 2];
        float ls[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] = 0.f;
#pragma unroll
        for (int e = 0; e < HB; e += 2) {
          const float p0 = ptx::ex2(fmaf(s[e], cs, -m_use));
          const float p1 = ptx::ex2(fmaf(s[e + 1], cs, -m_use));
          ls[(e >> 1) & 7] += p0 + p1;
          pk[e / 2] = pack2(p0, p1, BF16);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));

        // O may be rescaled once the previous P.V product of this piece has
        // completed (the previous piece's epilogue waited for its own).  The
        // wait is taken on every tile so that this barrier's phases stay within
        // one of the waiter's (a parity wait cannot tell phase k from k + 2).
        if (j > 0 && alive)
          alive = __all_sync(0xffffffffu, wait_bar(bar(kBarPvDone), (gt - 1) & 1, abort_flag,
                                                   p.status, kDevTimeoutPvDone));
        // A warp whose wait gave up skips the rest of the tile; it stops together
        // with its partner at the next swap.
        if (!alive) continue;
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float a = rescale_o ? alpha : 1.f;
#pragma unroll 1
          for (int cch = 0; cch < C::DV / 64; ++cch) {
            const uint32_t col = half * (C::DV / 2) + cch * 32;
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + col, r);
            ptx::tmem_wait_ld();
            ptx::reg_fence(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a);
            ptx::tmem_st32(lane_base + col, r);
          }
          ptx::tmem_wait_st();
        }
        if constexpr (C::PSM) {
          // P row -> shared memory, K-major 128B-swizzled (64 keys per 128-byte row).
#pragma unroll
          for (int ch = 0; ch < HB / 8; ++ch) {
            const int gc = half * (HB / 8) + ch;
            const int blk = gc >> 3, cc = gc & 7;
            const uint32_t addr = sP + blk * 16384 + t * 128 + ((cc ^ (t & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * ch]),
                         "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                         : "memory");
          }
          ptx::fence_proxy_async_smem();
        } else {
          // P row -> tensor memory, over the first BN/2 columns of the S buffer
          // it came from (two 16-bit probabilities per column; this thread's
          // keys at columns [half * HB/2, (half + 1) * HB/2)).  The other half of
          // the row has read its S columns: both passed the row-max swap.
          const uint32_t pcol = lane_base + C::S_COL + buf * BN + half * (HB / 2);
          if constexpr (HB == 64)
            ptx::tmem_st32(pcol, pk);
          else
            ptx::tmem_st16(pcol, pk);
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        warp_arrive(kBarPFull);
      }
      if (ok && count > 0) {
        if (alive)
          alive = __all_sync(0xffffffffu, wait_bar(bar(kBarPvDone), (g0 + count - 1) & 1,
                                                   abort_flag, p.status, kDevTimeoutPvDone));
        ptx::tc_fence_after();
        float lo = 0.f;
        ok = swap_half(l, lo);
        l = half == 0 ? l + lo : lo + l;  // both halves: l_0 + l_1
      }
      // All 256 threads take the epilogue, with its CTA-wide barriers, or none.
      ok = ptx::bar_red_and(1, 256, ok);
      if (!ok) break;
      // -------------------------------------------------------------- epilogue
      const long long R = static_cast<long long>(p.B) * p.Hq * p.Lq;
      // Suffix slot `sl` of this CTA: (max, sum) per row, and the 256 fp32 columns
      // as 64 groups of 4, each group stored for all 128 rows in a row, so that a
      // warp's float4 accesses to one group cover 512 contiguous bytes.
      auto sk_row = [&](int sl) -> long long {
        return (static_cast<long long>(sl) * 2 + rank) * 128 + t;
      };
      auto sk_o4 = [&](int sl, int c4) -> float4* {
        return reinterpret_cast<float4*>(p.sk_o) +
               ((static_cast<long long>(sl) * 2 + rank) * 64 + c4) * 128 + t;
      };
      if (C::DEC && pc.kind == 3) {
        // Cluster split: (max, sum) of every row into the idle query buffer and
        // the fp32 O rows into the idle ring (every load has been consumed and
        // every MMA has completed), for the cluster merge at the end.  Row t's
        // 16-byte chunk c sits at chunk c ^ (t & 15) of its DV * 4-byte row.
        if (count == 0) {
          // The query copies issued at entry were never waited for: let every
          // one of them land before the query buffer is reused.
          ptx::cp_async_wait_all();
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
        if (half == 0) reinterpret_cast<float2*>(smem + C::Q_OFF)[t] = make_float2(m_run, l);
        if (count > 0) {
#pragma unroll 1
          for (int cch = 0; cch < C::DV / 64; ++cch) {
            const int col = half * (C::DV / 2) + cch * 32;
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + col, r);
            ptx::tmem_wait_ld();
            ptx::reg_fence(r);
            if (row_valid) {
              const uint32_t rowa = sbase + C::RING_OFF + static_cast<uint32_t>(t * C::DV * 4);
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const uint32_t ci = static_cast<uint32_t>((col >> 2) + g) ^ static_cast<uint32_t>(t & 15);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rowa + (ci << 4)),
                             "r"(r[4 * g]), "r"(r[4 * g + 1]), "r"(r[4 * g + 2]), "r"(r[4 * g + 3])
                             : "memory");
              }
            }
          }
        }
      } else if (pc.kind == 3) {
        // Planned split: fp32 partials merged by the combine kernel.
        if (row_valid && half == 0 && (!PAIR || rank == 0)) {
          const long long pr = static_cast<long long>(w.split) * R + row_id;
          p.part_ml[2 * pr] = m_run;
          p.part_ml[2 * pr + 1] = l;
        }
        if (count > 0) {
#pragma unroll 1
          for (int cch = 0; cch < C::DV / 64; ++cch) {
            const int col = half * (C::DV / 2) + cch * 32;
            uint32_t r[32];
            ptx::tmem_ld32(lane_base + col, r);
            ptx::tmem_wait_ld();
            ptx::reg_fence(r);
            if (row_valid) {
              float4* dst = reinterpret_cast<float4*>(
                  p.part_o + (static_cast<long long>(w.split) * R + row_id) * p.D + d0 + col);
#pragma unroll
              for (int g = 0; g < 8; ++g)
                dst[g] = make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                     __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
            }
          }
        }
      } else if (C::DEC) {
        // (decode pieces are always cluster splits)
      } else if (pc.kind == 2) {
        // Suffix piece: leave the unnormalised share for the unit that holds the
        // query tile's prefix, then publish it.
        const long long sr = sk_row(pc.slot);
        if (half == 0) reinterpret_cast<float2*>(p.sk_ml)[sr] = make_float2(m_run, l);
#pragma unroll 1
        for (int cch = 0; cch < C::DV / 64; ++cch) {
          const int col = half * (C::DV / 2) + cch * 32;
          uint32_t r[32];
          ptx::tmem_ld32(lane_base + col, r);
          ptx::tmem_wait_ld();
          ptx::reg_fence(r);
#pragma unroll
          for (int g = 0; g < 8; ++g)
            *sk_o4(pc.slot, col / 4 + g) =
                make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                            __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3]));
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");
        if (threadIdx.x == 0 && p.withhold_q != 2) {
          __threadfence();
          asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p.sk_flag + pc.slot * 2 + rank),
                       "l"(p.epoch)
                       : "memory");
        }
      } else if (count > 0) {
        // Whole query tile (kind 0) or prefix (kind 1): merge the suffix shares,
        // if any, in key order, then normalise and store.
        int n_contrib = pc.kind == 1 ? pc.n_contrib : 0;
        if (n_contrib > 0) {
          if (threadIdx.x == 0) {
            for (int k = 0; k < n_contrib; ++k) {
              const unsigned long long* f = p.sk_flag + (pc.slot + k) * 2 + rank;
              const uint64_t t0 = ptx::globaltimer();
              for (uint32_t it2 = 0;; ++it2) {
                unsigned long long v;
                asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
                if (v == p.epoch) break;
                if ((it2 & 63) == 63 && (*abort_flag || ptx::globaltimer() - t0 > kTimeoutNs)) {
                  *abort_flag = 1;
                  atomicCAS(p.status, 0, kDevTimeoutPair);
                  break;
                }
              }
            }
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
        // A wait for the suffix shares that gave up (or any other abort of this
        // CTA) leaves them unknown: merge nothing and store NaN rows, so that a
        // caller who skips the status check cannot take the tile for a result.
        const bool poisoned = n_contrib > 0 && *abort_flag != 0;
        if (poisoned) n_contrib = 0;
        // Combined max and sum (fixed order: own share, then units in order).
        float mtot = m_run;
        for (int k = 0; k < n_contrib; ++k) {
          const float2 mlk = __ldcg(reinterpret_cast<const float2*>(p.sk_ml) + sk_row(pc.slot + k));
          if (mlk.y > 0.f) mtot = fmaxf(mtot, mlk.x);
        }
        const float a_own = n_contrib == 0 ? 1.f : (l > 0.f ? ptx::ex2(m_run - mtot) : 0.f);
        float ltot = a_own * l;
        for (int k = 0; k < n_contrib; ++k) {
          const float2 mlk = __ldcg(reinterpret_cast<const float2*>(p.sk_ml) + sk_row(pc.slot + k));
          if (mlk.y > 0.f) ltot += ptx::ex2(mlk.x - mtot) * mlk.y;
        }
        const float inv = poisoned ? __int_as_float(0x7fc00000) : (ltot > 0.f ? 1.f / ltot : 0.f);
#pragma unroll 1
        for (int cch = 0; cch < C::DV / 64; ++cch) {
          const int col = half * (C::DV / 2) + cch * 32;
          uint32_t r[32];
          ptx::tmem_ld32(lane_base + col, r);
          ptx::tmem_wait_ld();
          ptx::reg_fence(r);
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]) * a_own;
          for (int k = 0; k < n_contrib; ++k) {
            const long long sr = sk_row(pc.slot + k);
            const float2 mlk = __ldcg(reinterpret_cast<const float2*>(p.sk_ml) + sr);
            if (!(mlk.y > 0.f)) continue;
            const float ak = ptx::ex2(mlk.x - mtot);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const float4 v = __ldcg(sk_o4(pc.slot + k, col / 4 + g));
              o[4 * g] = fmaf(ak, v.x, o[4 * g]);
              o[4 * g + 1] = fmaf(ak, v.y, o[4 * g + 1]);
              o[4 * g + 2] = fmaf(ak, v.z, o[4 * g + 2]);
              o[4 * g + 3] = fmaf(ak, v.w, o[4 * g + 3]);
            }
          }
          if constexpr (C::STAGE) {
            // Through this warp's 4 KB slice of the P buffer (with Q in TMEM, P's
            // last product has completed; otherwise the buffer holds nothing
            // else): 32 rows x 64 columns a round, written row-wise and
            // read back so that one global store covers four whole 128-byte
            // lines.  Chunk c of slice row r sits at 16-byte position c ^ (r & 7).
            const uint32_t slice = sP + static_cast<uint32_t>(warp) * 4096u;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 v;
              v.x = pack2(o[8 * g + 0] * inv, o[8 * g + 1] * inv, BF16);
              v.y = pack2(o[8 * g + 2] * inv, o[8 * g + 3] * inv, BF16);
              v.z = pack2(o[8 * g + 4] * inv, o[8 * g + 5] * inv, BF16);
              v.w = pack2(o[8 * g + 6] * inv, o[8 * g + 7] * inv, BF16);
              const int cc = (cch & 1) * 4 + g;
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               slice + lane * 128 + ((cc ^ (lane & 7)) << 4)),
                           "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                           : "memory");
            }
            if (cch & 1) {
              __syncwarp();
              const int colr = col - 32;  // first column of this 64-column round
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const int rr = 4 * k + (lane >> 3);  // slice row
                const int c = lane & 7;
                uint4 v;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                             : "r"(slice + rr * 128 + ((c ^ (rr & 7)) << 4))
                             : "memory");
                const int i = w.m0 + q4 * 32 + rr;  // query row of slice row rr
                if (i < p.Lq) {
                  const long long rid = (static_cast<long long>(w.b) * p.Hq + w.h0) * p.Lq + i;
                  *reinterpret_cast<uint4*>(p.out + rid * p.D + d0 + colr + c * 8) = v;
                }
              }
              __syncwarp();  // the slice is rewritten by the next round
            }
          } else if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + row_id * p.D + d0 + col);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              uint4 v;
              v.x = pack2(o[8 * g + 0] * inv, o[8 * g + 1] * inv, BF16);
              v.y = pack2(o[8 * g + 2] * inv, o[8 * g + 3] * inv, BF16);
              v.z = pack2(o[8 * g + 4] * inv, o[8 * g + 5] * inv, BF16);
              v.w = pack2(o[8 * g + 6] * inv, o[8 * g + 7] * inv, BF16);
              dst[g] = v;
            }
          }
        }
      }
      if (count > 0) {
        // This piece's reads of O are complete: the next piece may overwrite it.
        ptx::tc_fence_before();
        warp_arrive(kBarOFree);
      }
      g0 += count;
    }
    if constexpr (C::DEC) {
      // Cluster merge.  Every CTA (split) of the cluster has left (max, sum)
      // per row in its query buffer and its fp32 O rows in its ring.  CTA
      // `crank` merges output columns [crank * DV / CS, (crank + 1) * DV / CS)
      // of every row over the CS splits in rank order:
      //   M = max_s m_s,  L = sum_s 2^(m_s - M) l_s,  O = sum_s 2^(m_s - M) O_s,
      // skipping splits that saw no visible key (l_s == 0), and stores O / L
      // (one cluster per group) or (M, L, O) as this cluster's partial for the
      // combine kernel.  A row's result depends on that row's partials only.
      // If any CTA of the cluster gave up a wait, the merged rows are NaN.  The
      // producer / MMA warpgroup takes part in the two cluster barriers.
      ptx::cp_async_wait_all();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      ptx::cluster_sync();  // all partials and abort flags of the cluster are in place
      const int CS = p.dec_cs;
      const uint32_t crank = ptx::cluster_ctarank();
      // The abort flags are requested here and tested after the partials'
      // loads have been issued, so that both cost one round trip.
      uint32_t aborted[kMaxDecodeClusterCtas];
#pragma unroll
      for (int r = 0; r < kMaxDecodeClusterCtas; ++r)
        aborted[r] = r < CS ? ptx::ld_cluster_u32(ptx::mapa(sbase + C::BAR_OFF + 244, r)) : 0u;
      const Work w = make_work<BN, QROWS>(p, item, 0);
      const int ncol = C::DV / CS;
      const int nch = ncol >> 2;
      const int c0 = static_cast<int>(crank) * ncol;
      const int base = p.Lk - p.Lq;
      const long long R = static_cast<long long>(p.B) * p.Hq * p.Lq;
      const int cl = w.split / CS;  // this cluster's index within its group
      const float qnan = __int_as_float(0x7fc00000);
      for (int idx = threadIdx.x; idx < 128 * nch; idx += 256) {
        const int tt = idx / nch, ch = idx - tt * nch;
        const int hl = tt >> 3;
        const int i = ((((tt & 7) - base) % 8) + 8) % 8;
        const int h = w.h0 + hl;
        if (!(i < p.Lq && hl < min(p.G, 16) && h < (w.hkv + 1) * p.G)) continue;
        const long long row_id = (static_cast<long long>(w.b) * p.Hq + h) * p.Lq + i;
        const uint32_t mla = sbase + C::Q_OFF + static_cast<uint32_t>(tt * 8);
        const uint32_t ci = static_cast<uint32_t>((c0 >> 2) + ch) ^ static_cast<uint32_t>(tt & 15);
        const uint32_t oa = sbase + C::RING_OFF + static_cast<uint32_t>(tt * C::DV * 4) + (ci << 4);
        // All loads first (issued back to back), then the arithmetic.
        float2 ml[kMaxDecodeClusterCtas];
        float4 o[kMaxDecodeClusterCtas];
#pragma unroll
        for (int r = 0; r < kMaxDecodeClusterCtas; ++r)
          if (r < CS) ml[r] = ptx::ld_cluster_f2(ptx::mapa(mla, r));
#pragma unroll
        for (int r = 0; r < kMaxDecodeClusterCtas; ++r)
          if (r < CS) o[r] = ptx::ld_cluster_f4(ptx::mapa(oa, r));
        bool bad = false;
#pragma unroll
        for (int r = 0; r < kMaxDecodeClusterCtas; ++r) bad |= aborted[r] != 0u;
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxDecodeClusterCtas; ++r)
          if (r < CS && ml[r].y > 0.f) M = fmaxf(M, ml[r].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kMaxDecodeClusterCtas; ++r) {
          if (r < CS && ml[r].y > 0.f) {
            const float wgt = ptx::ex2(ml[r].x - M);
            L = fmaf(wgt, ml[r].y, L);
            acc.x = fmaf(wgt, o[r].x, acc.x);
            acc.y = fmaf(wgt, o[r].y, acc.y);
            acc.z = fmaf(wgt, o[r].z, acc.z);
            acc.w = fmaf(wgt, o[r].w, acc.w);
          }
        }
        const int col = c0 + 4 * ch;
        if (p.dec_nc == 1) {
          const float inv = bad ? qnan : (L > 0.f ? 1.f / L : 0.f);
          uint2 v;
          v.x = pack2(acc.x * inv, acc.y * inv, BF16);
          v.y = pack2(acc.z * inv, acc.w * inv, BF16);
          *reinterpret_cast<uint2*>(p.out + row_id * p.D + col) = v;
        } else {
          if (bad) acc = make_float4(qnan, qnan, qnan, qnan);
          const long long pr = static_cast<long long>(cl) * R + row_id;
          *reinterpret_cast<float4*>(p.part_o + pr * p.D + col) = acc;
          if (crank == 0 && ch == 0)
            reinterpret_cast<float2*>(p.part_ml)[pr] = make_float2(M, bad ? qnan : L);
        }
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // (re)converge before the aligned barrier
      // This CTA has read what it needs from the others' shared memory; the
      // matching wait, before any CTA of the cluster exits, is at teardown.
      ptx::cluster_arrive();
    }
  }

  // ------------------------------------------------------------------ teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Let every copy and MMA this CTA started finish before its memory goes away.
    if (warp == C::kProducerWarp && lane == 0) {
      if (issued_q && mma_cta)
        wait_bar(bar(kBarQ), (issued_q - 1) & 1, abort_flag, p.status, kDevTimeoutDrain);
      for (int s = 0; s < C::NSLOT; ++s)
        if (static_cast<uint32_t>(s) < ring_issued && mma_cta) {
          // the most recent load into slot s had sequence number `last`
          const uint32_t last = s + ((ring_issued - 1 - s) / C::NSLOT) * C::NSLOT;
          const uint32_t ph = (last / C::NSLOT) & 1;
          const uint64_t t0 = ptx::globaltimer();
          while (!ptx::mbar_try_wait(bar(kBarKvFull + s), ph) &&
                 ptx::globaltimer() - t0 < kTimeoutNs) {
          }
        }
    }
    if (warp == C::kMmaWarp && lane == 0 && mma_issued) {
      if constexpr (DUO)
        ptx::mma_commit_pair_mc(bar(kBarDrain), 1);
      else
        ptx::mma_commit(bar(kBarDrain));
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(bar(kBarDrain), 0) && ptx::globaltimer() - t0 < kTimeoutNs) {
      }
    }
    __syncthreads();
  }
  // The peer may still write into our shared memory (PAIR) or read our tiles and
  // tensor memory through 2-SM MMAs (DUO) until both CTAs get here.
  if (CLUSTER) ptx::cluster_sync();
  // Decode: the other CTAs of the cluster may still read this one's partials
  // until all of them have arrived after the merge.
  if (C::DEC) ptx::cluster_wait();
  if (warp == C::kMmaWarp) {
    ptx::tc_fence_after();
    if constexpr (DUO)
      ptx::tmem_dealloc_pair(tmem, 512);
    else
      ptx::tmem_dealloc(tmem, 512);
  }
}


// Merge split partials: for each row, M = max_s m_s, l = sum_s 2^(m_s - M) l_s,
// out = sum_s 2^(m_s - M) O_s / l, splits that saw no visible key (l_s == 0)
// skipped and a poisoned split (l_s NaN) carried into the row.  Grid (rows,
// ceil(D / 128)); 256 threads.  Every warp finds M (a warp-shuffle maximum,
// exact in any order); warp w accumulates splits w, w+8, w+16, ... for 128
// columns (4 per lane), and the eight warp sums of O and l are added in warp
// order.  Every sum runs in a
// fixed order, so a row's result depends only on that row's partials.
constexpr int kCombineThreads = 256;

template <bool BF16>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_ml,
    uint16_t* __restrict__ out, long long R, int D, int n_splits) {
  __shared__ float4 acc_w[8][32];
  __shared__ float l_w[8];
  // Launched as a programmatic dependent of the attention grid: wait until that
  // grid has completed and its partials are visible.
  ptx::griddep_wait();
  const long long row = blockIdx.x;
  const int c0 = blockIdx.y * 128;
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const bool col_ok = c0 + 4 * lane < D;  // head_dim 192: the second block is half full
  const float2* ml_row = reinterpret_cast<const float2*>(part_ml) + row;
  const float* base = part_o + row * D + c0 + 4 * lane;
  const long long split_stride = R * D;
  // Warp w takes splits w, w + 8, w + 16, ..., U of them a round; the first
  // round's loads are issued before those of the maximum, so that up to 8U
  // splits cost one round trip to memory.
  constexpr int U = 16;
  float4 v[U];
  float2 ml[U];
  auto load_round = [&](int s0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = s0 + 8 * u;
      ml[u] = s < n_splits ? ml_row[s * R] : make_float2(0.f, 0.f);
      v[u] = (s < n_splits && col_ok) ? *reinterpret_cast<const float4*>(base + s * split_stride)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  load_round(warp);
  float mx = -INFINITY;
#pragma unroll 4
  for (int s = lane; s < n_splits; s += 32) {
    const float2 m = ml_row[s * R];
    if (m.y > 0.f) mx = fmaxf(mx, m.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  for (int s0 = warp;;) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!(ml[u].y <= 0.f)) {  // saw a key, or poisoned (NaN)
        const float wv = ptx::ex2(ml[u].x - mx);
        a.x = fmaf(wv, v[u].x, a.x);
        a.y = fmaf(wv, v[u].y, a.y);
        a.z = fmaf(wv, v[u].z, a.z);
        a.w = fmaf(wv, v[u].w, a.w);
        lsum = fmaf(wv, ml[u].y, lsum);
      }
    }
    s0 += 8 * U;
    if (s0 >= n_splits) break;
    load_round(s0);
  }
  acc_w[warp][lane] = a;
  if (lane == 0) l_w[warp] = lsum;
  __syncthreads();
  if (warp == 0) {
    float4 sum = acc_w[0][lane];
    float lt = l_w[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      const float4 b = acc_w[w][lane];
      sum.x += b.x;
      sum.y += b.y;
      sum.z += b.z;
      sum.w += b.w;
      lt += l_w[w];
    }
    const float inv = lt > 0.f ? 1.f / lt : (lt == lt ? 0.f : lt);
    uint2 o;
    o.x = pack2(sum.x * inv, sum.y * inv, BF16);
    o.y = pack2(sum.z * inv, sum.w * inv, BF16);
    if (col_ok) *reinterpret_cast<uint2*>(out + row * D + c0 + 4 * lane) = o;
  }
}

}  // namespace gbsdpa
