// sdpa_api.cu -- host side of libsdpa_gb300.so: argument validation, TMA
// descriptor encoding, work planning and launches.  The C ABI is declared in
// include/sdpa_gb300.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <cstdint>
#include <mutex>

#include "sdpa_gb300.h"
#include "sdpa_launch.cuh"

namespace {

using gbsdpa::AttnParams;
using gbsdpa::Cfg;
using gbsdpa_host::DeviceState;

__device__ int g_device_status;

constexpr int kMaxDevices = 64;


std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SDPA_ERR_CUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return SDPA_ERR_CUDA;
    st.status = static_cast<int*>(addr);
    // Suffix-piece flags hold the epoch of the launch that wrote them.  Start from a
    // clock-derived value so that a workspace left over from another process
    // can never hold the epoch of a launch of this one.
    const auto now = std::chrono::steady_clock::now().time_since_epoch().count();
    st.epoch = (static_cast<unsigned long long>(now) * 0x9E3779B97F4A7C15ull) >> 1;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return SDPA_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return SDPA_OK;
}

// 3-D map over a contiguous [BH, L, D] tensor: dims (D, L, BH), box (64, rows, 1),
// 128-byte swizzle; rows past L read as zero and never spill into the next head.
int encode_map(CUtensorMap* m, const void* base, int D, long long L, long long BH, int rows,
               bool bf16, long long plane_rows = 0) {
  // plane_rows: rows from one (b, h) plane to the next (L for a packed tensor;
  // a K/V cache's capacity otherwise).
  if (plane_rows <= 0) plane_rows = L;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                           static_cast<cuuint64_t>(plane_rows) * static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SDPA_OK : SDPA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head_dim(int D) { return D == 128 || D == 192 || D == 256 || D == 512; }

int validate(const void* q, const void* k, const void* v, const void* out, int B, int Hq, int Hkv,
             int Lq, int Lk, int D, float scale, int causal, int window, int dtype) {
  if (!q || !k || !v || !out) return SDPA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0) return SDPA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SDPA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SDPA_ERR_INVALID_ARG;
  if (window < 0 || (window > 0 && !causal)) return SDPA_ERR_INVALID_ARG;
  if (causal && Lq > Lk) return SDPA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return SDPA_ERR_INVALID_ARG;
  if (!supported_head_dim(D)) return SDPA_ERR_UNSUPPORTED;
  if (dtype != SDPA_F16 && dtype != SDPA_BF16) return SDPA_ERR_UNSUPPORTED;
  // TMA coordinates and flat row indices stay within 32-bit / 64-bit ranges.
  if (static_cast<long long>(B) * Hq > (1ll << 30) || static_cast<long long>(B) * Hkv > (1ll << 30))
    return SDPA_ERR_INVALID_ARG;
  if (Lk > (1 << 30) || Lq > (1 << 30)) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SDPA_ERR_ALIGNMENT;
  return SDPA_OK;
}

// K/V in a cache of kv_cap rows per (b, kv head): packed rows 0..Lk-1
// (kv_cap >= Lk), or a ring where key j sits in row j mod kv_cap.  A ring must
// hold every key some row can see (the window plus the query rows, or all Lk
// keys without a window) and a multiple of 128 rows, so that no key tile wraps.
// Head dims: Q/K and V equal (128, 192, 256, 512), or Q/K 192 with V 256.
int validate_dims(int Dqk, int Dv) {
  if (Dqk == Dv) return SDPA_OK;  // checked with the rest of the arguments
  return (Dqk == 192 && Dv == 256) ? SDPA_OK : SDPA_ERR_UNSUPPORTED;
}

// Additive bias: entry (b, h, i, j) at ptr[b * sb + h * sh + i * sq + j], in q's
// dtype; strides are elements, >= 0 (0 broadcasts).  Null ptr: no bias.
struct BiasArg {
  const void* ptr = nullptr;
  long long sb = 0, sh = 0, sq = 0;
};

int validate_bias(const BiasArg& b) {
  if (!b.ptr) return SDPA_OK;
  const long long lim = 1ll << 48;
  if (b.sb < 0 || b.sh < 0 || b.sq < 0 || b.sb > lim || b.sh > lim || b.sq > lim)
    return SDPA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(b.ptr) & 1u) return SDPA_ERR_ALIGNMENT;
  return SDPA_OK;
}

int validate_kv_layout(int Lq, int Lk, int causal, int window, int kv_cap, int kv_ring) {
  if (kv_ring != 0 && kv_ring != 1) return SDPA_ERR_INVALID_ARG;
  if (kv_cap <= 0 || kv_cap > (1 << 30)) return SDPA_ERR_INVALID_ARG;
  if (!kv_ring) return kv_cap >= Lk ? SDPA_OK : SDPA_ERR_INVALID_ARG;
  if (kv_cap % 128 != 0) return SDPA_ERR_INVALID_ARG;
  const long long span = (causal && window > 0)
                             ? std::min<long long>(Lk, static_cast<long long>(Lq) + window - 1)
                             : Lk;
  return span <= kv_cap ? SDPA_OK : SDPA_ERR_INVALID_ARG;
}

int launch_combine(const float* part_o, const float* part_ml, void* out, long long R, int D,
                   int n_splits, bool bf16, cudaStream_t stream) {
  if (R <= 0 || R > 0x7fffffffll || D % 64 != 0) return SDPA_ERR_INVALID_ARG;
  // Programmatic dependent launch: the merge grid's CTAs may be placed while the
  // attention grid drains; the kernel waits for that grid before reading.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(R), static_cast<unsigned>((D + 127) / 128));
  cfg.blockDim = dim3(gbsdpa::kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint16_t* o = static_cast<uint16_t*>(out);
  const cudaError_t e =
      bf16 ? cudaLaunchKernelEx(&cfg, gbsdpa::combine_kernel<true>, part_o, part_ml, o, R, D, n_splits)
           : cudaLaunchKernelEx(&cfg, gbsdpa::combine_kernel<false>, part_o, part_ml, o, R, D, n_splits);
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

size_t partial_bytes(long long R, int D, int n_splits) {
  // part_o then part_ml, each 256-byte aligned.
  const size_t po = static_cast<size_t>(n_splits) * static_cast<size_t>(R) * D * sizeof(float);
  const size_t pm = static_cast<size_t>(n_splits) * static_cast<size_t>(R) * 2 * sizeof(float);
  return ((po + 255) & ~static_cast<size_t>(255)) + ((pm + 255) & ~static_cast<size_t>(255));
}

// Kernel variant for a call: head_dim 512 splits the head dimension over a CTA
// pair; head_dim 256 and 128 prefill use 2-SM MMAs over 256-row query tiles (a
// 2-SM tile costs about two thirds of two 1-SM tiles), except with a sliding
// window shorter than 256 keys, where most of a 256-row tile's keys would be
// masked; head_dim 192 prefill stays on one CTA (the 2-SM tile would split V
// into 96-column halves, which a 128-byte-swizzled 64-column box cannot hold);
// decode uses one CTA per 16 query heads x 8 position slots and split, the
// splits of a head group forming a cluster (kDecode) below head_dim 512.
int choose_mode(bool decode, int D, int window) {
  if (D == 512) return decode ? gbsdpa::kPairXD : gbsdpa::kPairX;
  if (decode) return gbsdpa::kDecode;
  if (D == 192) return gbsdpa::kSingle;
  return (window > 0 && window < 256) ? gbsdpa::kSingle : gbsdpa::kDuo;
}


// The instantiation a call of this shape launches: at head dim 256 without a
// bias the 2-SM variant keeps Q in tensor memory (measured faster over long
// key ranges, and, with head-paired tiles, over a sliding window's short
// pieces; a bias's loads do better with the form that keeps P in tensor
// memory).
int launch_mode(int mode, int D, int Dv, int window, bool bias) {
  (void)window;
  return (mode == gbsdpa::kDuo && D == 256 && Dv == 256 && !bias) ? gbsdpa::kDuoQ : mode;
}

bool two_sm(int mode) { return mode == gbsdpa::kDuo || mode == gbsdpa::kDuoQ; }
// Query-tile geometry of a prefill call: rows per tile and query heads per work
// item.  A 2-SM pair takes 128 rows of two query heads of one kv head when the
// group size is even (both CTAs then see the same key band: a sliding window
// spans window + 127 keys instead of window + 255), else 256 rows of one head.
struct QTiling {
  int rows = 128, heads = 1;
};
QTiling qtiling(int mode, int G) {
  QTiling t;
  if (two_sm(mode)) {
    if (G % 2 == 0)
      t.heads = 2;
    else
      t.rows = 256;
  }
  return t;
}
int key_tile(int mode) {
  return (mode == gbsdpa::kPairX || mode == gbsdpa::kPairXD || mode == gbsdpa::kDecode) ? 64
                                                                                       : 128;
}

// Key tiles the longest query tile (of `rows` rows) visits.
long long max_tiles_per_qtile(int Lq, int Lk, int causal, int window, int bn, int rows) {
  if (!causal) return (Lk + bn - 1) / bn;
  const int q0 = ((Lq - 1) / rows) * rows;  // the last query tile sees the most keys
  const int pmin = Lk - Lq + q0, pmax = Lk - 1;
  const int lo = window ? std::max(0, pmin - window + 1) : 0;
  const int hi = std::min(Lk, pmax + 1);
  return (hi + bn - 1) / bn - lo / bn;
}

// How many contiguous shares to cut each query tile's key range into.  A
// simple wave model: time ~ ceil(ctas / sms) * ceil(tiles / s), plus the cost
// of writing and re-reading the fp32 partials.
int plan_prefill_splits(int sms, int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal,
                        int window) {
  const int mode = choose_mode(false, D, causal ? window : 0);
  const QTiling qt = qtiling(mode, Hq / Hkv);
  const int bn = key_tile(mode), rows = qt.rows;
  const long long items = static_cast<long long>(B) * (Hq / qt.heads) * ((Lq + rows - 1) / rows);
  const long long per_cta = mode == gbsdpa::kSingle ? 1 : 2;
  const long long slots = std::max<long long>(1, sms / per_cta);
  const long long T = max_tiles_per_qtile(Lq, Lk, causal, window, bn, rows);
  if (items >= 2 * slots || T < 16) return 1;
  // one key tile ~ 4 * 128 * bn * 256 flop per CTA at ~8 Kflop/clk, ~1.9 GHz
  const double t_tile_us = 4.0 * 128 * bn * 256 / 8192.0 / 1900.0;
  const double partial_us_per_split =
      static_cast<double>(B) * Hq * Lq * D * 4.0 * 2.0 / 6.0e6;  // write + read at ~6 TB/s
  int best = 1;
  double best_t = 1e300;
  for (int s = 1; s <= 8; ++s) {
    const long long waves = (items * s + slots - 1) / slots;
    const double t = waves * ((T + s - 1) / s) * t_tile_us + (s > 1 ? s * partial_us_per_split : 0);
    if (t < best_t * 0.97) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

int plan_decode_splits(int sms, int B, int Hq, int Hkv, int D, int window = 0) {
  const int G = Hq / Hkv;
  const long long n_hb = (G + 15) / 16;
  const long long per_cta = D == 512 ? 2 : 1;
  const long long units = static_cast<long long>(B) * Hkv * n_hb * per_cta;
  long long s = sms / std::max<long long>(1, units);
  // A window reaches only about window / key-tile tiles: more splits than that
  // sit idle and still cost the merge (measured: 19 -> 10 splits takes the
  // head_dim-256 w1024 decode from 22.2 to 20.6 us).  The count depends on the
  // window, never on Lq or Lk, so row invariance is kept.
  if (window > 0) {
    const int bn = D == 512 ? 64 : 128;
    s = std::min<long long>(s, (window + bn - 1) / bn + 1);
  }
  s = std::max<long long>(1, std::min<long long>(s, 256));
  return static_cast<int>(s);
}

// Decode split plan.  S splits per (batch, kv head, head block) group deal the
// group's key tiles round-robin.  kDecode (head dim <= 256): the splits are NC
// clusters of CS CTAs (S = CS * NC); a cluster merges its splits through
// distributed shared memory, so with one cluster per group a single launch
// writes the output and needs no workspace.  Everything here depends on
// (B, Hq, Hkv, D, window) and the device only, never on Lq or Lk: the split a
// tile goes to, and so every row's arithmetic, is the same for a verify call
// and the single-row call over its trimmed keys.
struct DecodePlan {
  int S = 1, CS = 0, NC = 1;  // CS = 0: not a cluster plan (head-dim-split pair)
};

long long decode_groups(int B, int Hq, int Hkv) {
  return static_cast<long long>(B) * Hkv * ((Hq / Hkv + 15) / 16);
}

DecodePlan plan_decode(DeviceState* st, int B, int Hq, int Hkv, int D, int Dv, int window) {
  DecodePlan pl;
  if (choose_mode(true, D, 0) != gbsdpa::kDecode) {
    pl.S = plan_decode_splits(st->sms, B, Hq, Hkv, D, window);
    return pl;
  }
  const long long groups = decode_groups(B, Hq, Hkv);
  // 64-key tiles the rows of a group can see: at most window + 7 keys (Lq <= 8).
  const long long t_max = window > 0 ? (window + 6 + 63) / 64 + 1 : (1ll << 30);
  const long long cap = std::min<long long>(
      {gbsdpa::kMaxDecodeClusterCtas, t_max, std::max<long long>(1, st->sms / groups)});
  // The largest power-of-two cluster whose clusters for all groups can be
  // resident at once (a second wave would double the latency).
  int cs = 1;
  while (cs * 2 <= cap) cs *= 2;
  for (; cs > 1; cs /= 2)
    if (gbsdpa_host::decode_fit(D, Dv, st, cs) >= groups) break;
  const int fit = std::max(1, gbsdpa_host::decode_fit(D, Dv, st, cs));
  long long nc = std::min<long long>(st->sms / (groups * cs), t_max / cs);
  nc = std::min<long long>(nc, fit / std::max<long long>(1, groups));
  pl.CS = cs;
  pl.NC = static_cast<int>(std::max<long long>(1, std::min<long long>(nc, 64)));
  pl.S = pl.CS * pl.NC;
  return pl;
}

// Workspace of a decode call with this plan: the fp32 partials the combine
// kernel merges (0 when the clusters write the output).
size_t decode_partial_bytes(const DecodePlan& pl, long long R, int Dv) {
  if (pl.CS > 0) return pl.NC > 1 ? partial_bytes(R, Dv, pl.NC) : 0;
  return partial_bytes(R, Dv, pl.S);
}

// ----------------------------------------------------------- persistent plan
// Prefill with one CTA (or 2-SM pair) per query tile leaves SMs idle when the
// query tiles do not fill whole waves.  The persistent variant keeps one unit
// per resident slot: units take the query tiles in waves and then share out the
// leftover partial wave by key tiles (the schedule is spelled out beside the
// kernel's iterator).  Only the unit count is chosen here.

// Key tiles a query tile of `rows` rows starting at q0 visits (the kernel's
// item_tiles_for_qt).
long long qtile_key_tiles(int q0, int rows, int Lq, int Lk, int causal, int window, int bn) {
  const int qlast = std::min(q0 + rows, Lq) - 1;
  const int pmin = Lk - Lq + q0, pmax = Lk - Lq + qlast;
  const int lo = (causal && window) ? std::max(0, pmin - window + 1) : 0;
  const int hi = causal ? std::min(Lk, pmax + 1) : Lk;
  return (hi + bn - 1) / bn - lo / bn;
}

// Key tiles of all work items (each item: one query tile of `heads` heads).
long long total_key_tiles(int B, int Hq, int Lq, int Lk, int causal, int window, int bn, int rows,
                          int heads) {
  long long w = 0;
  for (int q0 = 0; q0 < Lq; q0 += rows) w += qtile_key_tiles(q0, rows, Lq, Lk, causal, window, bn);
  return w * B * (Hq / heads);
}

// Workspace of a persistent launch: per (slot, rank) 128 x 256 fp32 partial
// rows, 128 (max, sum) pairs and one flag.
struct SkLayout {
  size_t o_off, ml_off, flag_off, bytes;
};

SkLayout sk_layout(long long units) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SkLayout L;
  L.o_off = 0;
  L.ml_off = up(static_cast<size_t>(units) * 2 * 128 * 256 * sizeof(float));
  L.flag_off = L.ml_off + up(static_cast<size_t>(units) * 2 * 128 * 2 * sizeof(float));
  L.bytes = L.flag_off + up(static_cast<size_t>(units) * 2 * sizeof(unsigned long long));
  return L;
}

// Prefix length L of the leftover items of a persistent launch (their first L
// key tiles stay on one unit each, the rest is shared out), with the suffix
// total SS and suffix unit count US.  Costs are in key tiles: a piece boundary
// costs about kPieceCost (query reload, pipeline refill, partial write), the
// prefix unit's merge about kMergeCost.  L balances the prefix units against
// the suffix units, or is the longest leftover item (no split) when the split
// would not be shorter.
struct TailPlan {
  int L = 0, US = 0;
  long long SS = 0;
};

TailPlan plan_tail(long long units, int B, int Hq, int Lq, int Lk, int causal, int window, int bn,
                   int rows, int heads) {
  constexpr long long kPieceCost = 3, kMergeCost = 3;
  TailPlan t;
  const long long n_qtiles = (Lq + rows - 1) / rows;
  const long long n_per = static_cast<long long>(B) * (Hq / heads);
  const long long N = n_qtiles * n_per, U = units;
  const long long r = N % U, base = N - r;
  if (r == 0) return t;
  auto T = [&](long long i) {  // key tiles of leftover item i
    const long long qt = n_qtiles - 1 - (base + i) / n_per;
    return qtile_key_tiles(static_cast<int>(qt * rows), rows, Lq, Lk, causal, window, bn);
  };
  long long wt = 0, tmax = 0;
  for (long long i = 0; i < r; ++i) {
    wt += T(i);
    tmax = std::max(tmax, T(i));
  }
  long long L = (wt + kPieceCost * U - kMergeCost * (U - r) + U - 1) / U;
  L = std::max(1ll, std::min(L, tmax));
  long long ss = 0;
  for (long long i = 0; i < r; ++i) ss += std::max(0ll, T(i) - L);
  const long long us = std::min(U - r, ss);
  bool split = ss > 0 && us > 0;
  if (split) {
    const long long per_suffix = (ss + us - 1) / us + kPieceCost * ((r + us - 1) / us + 1);
    const long long cost = std::max(L + kMergeCost, per_suffix);
    split = cost * 100 < tmax * 97;
  }
  if (!split) {
    t.L = static_cast<int>(tmax);
    return t;
  }
  t.L = static_cast<int>(L);
  t.SS = ss;
  t.US = static_cast<int>(us);
  return t;
}

// Units for a persistent prefill launch (0: one CTA per query tile instead).
template <bool BF16>
long long persistent_units(DeviceState* st, int mode, int D, int B, int Hq, int Hkv, int Lq,
                           int Lk, int causal, int window, int Dv = 0, bool bias = false) {
  if (Dv <= 0) Dv = D;
  const int lm = launch_mode(mode, D, Dv, causal ? window : 0, bias);
  const int units = bias ? gbsdpa_host::resident_bias_variant(BF16, lm, D, Dv, st)
                         : gbsdpa_host::resident_variant<BF16, false>(lm, D, Dv, st);
  if (units <= 0) return 0;
  const QTiling qt = qtiling(mode, Hq / Hkv);
  const long long W =
      total_key_tiles(B, Hq, Lq, Lk, causal, window, key_tile(mode), qt.rows, qt.heads);
  return std::min<long long>(units, W);
}

template <bool BF16>
int run(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv, int Lq,
        int Lk, int D, float scale, int causal, int window, bool decode, int n_splits,
        bool write_partial, void* workspace, cudaStream_t stream, DeviceState* st,
        int withhold_q = 0, long long sk_units = 0, int kv_cap = 0, int kv_ring = 0, int Dv = 0,
        const BiasArg& bias = BiasArg(), const DecodePlan* dplan = nullptr) {
  // D is the Q/K head dim; Dv (0: the same) is V's and the output's.  Decode
  // takes its split plan from `dplan` (n_splits / write_partial are ignored).
  if (Dv <= 0) Dv = D;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  const int mode = choose_mode(decode, D, window);
  int n_partials = n_splits;  // fp32 partials per row for the combine kernel
  if (mode == gbsdpa::kDecode) {
    if (!dplan || dplan->CS < 1) return SDPA_ERR_INVALID_ARG;
    n_splits = dplan->S;
    n_partials = dplan->NC;
    write_partial = dplan->NC > 1;
    p.dec_cs = dplan->CS;
    p.dec_nc = dplan->NC;
  } else if (decode) {
    if (!dplan) return SDPA_ERR_INVALID_ARG;
    n_splits = n_partials = dplan->S;
    write_partial = true;
  }
  // K boxes: all keys of a tile (one CTA, 128-key tiles), or 64 keys (pair
  // kernels, decode); V boxes: 32 keys (one CTA, head-dim split) or 64 keys
  // (2-SM MMA).
  const int k_rows = mode == gbsdpa::kSingle ? 128 : 64;
  const int v_rows = two_sm(mode) ? 64 : 32;
  int rc = SDPA_OK;
  if (!decode) rc = encode_map(&p.tm_q, q, D, Lq, static_cast<long long>(B) * Hq, 128, BF16);
  if (rc) return rc;
  // K/V: Lk keys packed, or in a cache of kv_cap rows per plane (a ring keeps
  // all kv_cap rows live).
  if (kv_cap <= 0) kv_cap = Lk;
  const long long kv_rows = kv_ring ? kv_cap : Lk;
  rc = encode_map(&p.tm_k, k, D, kv_rows, static_cast<long long>(B) * Hkv, k_rows, BF16, kv_cap);
  if (rc) return rc;
  rc = encode_map(&p.tm_v, v, Dv, kv_rows, static_cast<long long>(B) * Hkv, v_rows, BF16, kv_cap);
  if (rc) return rc;
  p.kv_ring = kv_ring ? kv_cap : 0;
  const long long R = static_cast<long long>(B) * Hq * Lq;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  if (write_partial) {
    const size_t po = static_cast<size_t>(n_partials) * static_cast<size_t>(R) * Dv * sizeof(float);
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         ((po + 255) & ~static_cast<size_t>(255)));
  }
  p.status = st->status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.D = Dv;
  p.Dqk = D;
  p.causal = causal;
  p.window = window;
  // c = scale * log2(e), kept > 0 so that a masked score (-inf) maps to -inf;
  // scale == 0 becomes a tiny c, for which every visible weight is exactly 1.
  p.c = std::max(static_cast<float>(static_cast<double>(scale) * 1.4426950408889634), 1e-30f);
  p.decode = decode ? 1 : 0;
  if (bias.ptr) {
    p.bias = static_cast<const uint16_t*>(bias.ptr);
    p.bias_sb = bias.sb;
    p.bias_sh = bias.sh;
    p.bias_sq = bias.sq;
    p.bias_vec = aligned16(bias.ptr) && bias.sb % 8 == 0 && bias.sh % 8 == 0 && bias.sq % 8 == 0;
  }
  const QTiling qt = qtiling(mode, Hq / Hkv);
  p.hpair = qt.heads == 2 ? 1 : 0;
  p.n_qtiles = (Lq + qt.rows - 1) / qt.rows;
  p.n_splits = n_splits;
  p.n_hb = (p.G + 15) / 16;
  p.write_partial = write_partial ? 1 : 0;
  p.withhold_q = withhold_q;
  long long items;
  if (sk_units > 0) {
    const SkLayout L = sk_layout(sk_units);
    char* ws = static_cast<char*>(workspace);
    p.persistent = 1;
    p.n_units = static_cast<int>(sk_units);
    const TailPlan tp = plan_tail(sk_units, B, Hq, Lq, Lk, causal, window, key_tile(mode),
                                  qt.rows, qt.heads);
    p.tail_L = tp.L;
    p.tail_SS = tp.SS;
    p.tail_US = tp.US;
    p.sk_o = reinterpret_cast<float*>(ws + L.o_off);
    p.sk_ml = reinterpret_cast<float*>(ws + L.ml_off);
    p.sk_flag = reinterpret_cast<unsigned long long*>(ws + L.flag_off);
    {
      std::lock_guard<std::mutex> lk(g_mu);
      p.epoch = ++st->epoch;
    }
    items = sk_units;
  } else if (decode)
    items = static_cast<long long>(B) * Hkv * n_splits * p.n_hb;
  else
    items = static_cast<long long>(B) * (Hq / qt.heads) * p.n_qtiles * n_splits;
  const int lm = launch_mode(mode, D, Dv, window, p.bias != nullptr);
  rc = p.bias ? gbsdpa_host::launch_bias_variant(BF16, lm, D, Dv, p, items, stream, st)
              : gbsdpa_host::launch_variant<BF16, false>(lm, D, Dv, p, items, stream, st);
  if (rc) return rc;
  if (write_partial)
    rc = launch_combine(p.part_o, p.part_ml, out, R, Dv, n_partials, BF16, stream);
  return rc;
}

}  // namespace

extern "C" {

size_t sdpa_prefill_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal,
                                    int window) {
  DeviceState* st = nullptr;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Hq % Hkv) return 0;
  if (!supported_head_dim(D)) return 0;
  if (causal != 0 && causal != 1) return 0;
  if (window < 0 || (causal && Lq > Lk)) return 0;
  if (device_state(&st)) return 0;
  const int mode = choose_mode(false, D, causal ? window : 0);
  const long long u =
      std::max(persistent_units<false>(st, mode, D, B, Hq, Hkv, Lq, Lk, causal, window),
               persistent_units<true>(st, mode, D, B, Hq, Hkv, Lq, Lk, causal, window));
  if (u > 0) return sk_layout(u).bytes;
  const int s = plan_prefill_splits(st->sms, B, Hq, Hkv, Lq, Lk, D, causal, window);
  if (s <= 1) return 0;
  return partial_bytes(static_cast<long long>(B) * Hq * Lq, D, s);
}

int sdpa_prefill_launches(int B, int Hq, int Hkv, int Lq, int Lk, int D, int causal, int window,
                          size_t workspace_bytes) {
  // The same checks sdpa_prefill makes on sizes and flags (no pointers here).
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || Hq % Hkv) return SDPA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SDPA_ERR_INVALID_ARG;
  if (window < 0 || (window > 0 && !causal) || (causal && Lq > Lk)) return SDPA_ERR_INVALID_ARG;
  if (!supported_head_dim(D)) return SDPA_ERR_UNSUPPORTED;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  const int mode = choose_mode(false, D, window);
  const long long u = persistent_units<false>(st, mode, D, B, Hq, Hkv, Lq, Lk, causal, window);
  if (u > 0) return 1;  // persistent with the workspace, one CTA per tile without
  const int s = plan_prefill_splits(st->sms, B, Hq, Hkv, Lq, Lk, D, causal, window);
  return (s > 1 && workspace_bytes >= partial_bytes(static_cast<long long>(B) * Hq * Lq, D, s))
             ? 2 : 1;
}

size_t sdpa_decode_workspace_bytes(int B, int Hq, int Hkv, int Lq, int D) {
  DeviceState* st = nullptr;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lq > 8 || Hq % Hkv) return 0;
  if (!supported_head_dim(D)) return 0;
  if (device_state(&st)) return 0;
  // The plan without a window: a window never needs more (it can only cut the
  // cluster size, and then to one cluster per group).
  const long long R = static_cast<long long>(B) * Hq * Lq;
  return decode_partial_bytes(plan_decode(st, B, Hq, Hkv, D, D, 0), R, D);
}

static int prefill_impl(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                        int Hkv, int Lq, int Lk, int D, int Dv, float scale, int causal,
                        int window, int dtype, int kv_cap, int kv_ring, void* workspace,
                        size_t workspace_bytes, sdpa_stream_t stream,
                        const BiasArg& bias = BiasArg()) {
  int rc = validate(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, dtype);
  if (rc) return rc;
  rc = validate_dims(D, Dv);
  if (rc) return rc;
  rc = validate_kv_layout(Lq, Lk, causal, window, kv_cap, kv_ring);
  if (rc) return rc;
  rc = validate_bias(bias);
  if (rc) return rc;
  if (workspace && !aligned16(workspace)) return SDPA_ERR_ALIGNMENT;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  const bool bf16 = dtype == SDPA_BF16;
  auto strm = reinterpret_cast<cudaStream_t>(stream);
  const int mode = choose_mode(false, D, window);
  const bool has_bias = bias.ptr != nullptr;
  const long long u =
      bf16 ? persistent_units<true>(st, mode, D, B, Hq, Hkv, Lq, Lk, causal, window, Dv,
                                    has_bias)
           : persistent_units<false>(st, mode, D, B, Hq, Hkv, Lq, Lk, causal, window, Dv,
                                     has_bias);
  if (u > 0 && workspace && workspace_bytes >= sk_layout(u).bytes)
    return bf16 ? run<true>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, false, 1,
                            false, workspace, strm, st, 0, u, kv_cap, kv_ring, Dv, bias)
                : run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, false, 1,
                             false, workspace, strm, st, 0, u, kv_cap, kv_ring, Dv, bias);
  int s = u > 0 ? 1 : plan_prefill_splits(st->sms, B, Hq, Hkv, Lq, Lk, D, causal, window);
  if (s > 1 && (!workspace ||
                workspace_bytes < partial_bytes(static_cast<long long>(B) * Hq * Lq, Dv, s)))
    s = 1;
  return bf16 ? run<true>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, false, s,
                          s > 1, workspace, strm, st, 0, 0, kv_cap, kv_ring, Dv, bias)
              : run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, false, s,
                           s > 1, workspace, strm, st, 0, 0, kv_cap, kv_ring, Dv, bias);
}

static int decode_impl(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                       int Hkv, int Lq, int Lk, int D, int Dv, float scale, int causal,
                       int window, int dtype, int kv_cap, int kv_ring, void* workspace,
                       size_t workspace_bytes, sdpa_stream_t stream,
                       const BiasArg& bias = BiasArg()) {
  int rc = validate(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, dtype);
  if (rc) return rc;
  rc = validate_dims(D, Dv);
  if (rc) return rc;
  rc = validate_kv_layout(Lq, Lk, causal, window, kv_cap, kv_ring);
  if (rc) return rc;
  rc = validate_bias(bias);
  if (rc) return rc;
  if (Lq > 8) return SDPA_ERR_INVALID_ARG;
  if (workspace && !aligned16(workspace)) return SDPA_ERR_ALIGNMENT;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  const bool bf16 = dtype == SDPA_BF16;
  const DecodePlan pl = plan_decode(st, B, Hq, Hkv, D, Dv, causal ? window : 0);
  const size_t need = decode_partial_bytes(pl, static_cast<long long>(B) * Hq * Lq, Dv);
  if (need > 0 && (!workspace || workspace_bytes < need)) return SDPA_ERR_WORKSPACE;
  auto strm = reinterpret_cast<cudaStream_t>(stream);
  return bf16 ? run<true>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, true, 0,
                          true, workspace, strm, st, 0, 0, kv_cap, kv_ring, Dv, bias, &pl)
              : run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, true, 0,
                           true, workspace, strm, st, 0, 0, kv_cap, kv_ring, Dv, bias, &pl);
}

int sdpa_prefill(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                 int Lq, int Lk, int D, float scale, int causal, int window, int dtype,
                 void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  return prefill_impl(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, D, scale, causal, window, dtype, Lk, 0,
                      workspace, workspace_bytes, stream);
}

int sdpa_decode(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                int Lq, int Lk, int D, float scale, int causal, int window, int dtype,
                void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  return decode_impl(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, D, scale, causal, window, dtype, Lk, 0,
                     workspace, workspace_bytes, stream);
}

int sdpa_prefill_ex(const void* q, const void* k, const void* v, void* out, int B, int Hq,
                    int Hkv, int Lq, int Lk, int Dqk, int Dv, float scale, int causal, int window,
                    int dtype, int kv_capacity, int kv_ring, const void* bias,
                    long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                    void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  BiasArg b;
  b.ptr = bias;
  b.sb = bias_stride_b;
  b.sh = bias_stride_h;
  b.sq = bias_stride_q;
  return prefill_impl(q, k, v, out, B, Hq, Hkv, Lq, Lk, Dqk, Dv, scale, causal, window, dtype,
                      kv_capacity, kv_ring, workspace, workspace_bytes, stream, b);
}

int sdpa_decode_ex(const void* q, const void* k, const void* v, void* out, int B, int Hq, int Hkv,
                   int Lq, int Lk, int Dqk, int Dv, float scale, int causal, int window,
                   int dtype, int kv_capacity, int kv_ring, const void* bias,
                   long long bias_stride_b, long long bias_stride_h, long long bias_stride_q,
                   void* workspace, size_t workspace_bytes, sdpa_stream_t stream) {
  BiasArg b;
  b.ptr = bias;
  b.sb = bias_stride_b;
  b.sh = bias_stride_h;
  b.sq = bias_stride_q;
  return decode_impl(q, k, v, out, B, Hq, Hkv, Lq, Lk, Dqk, Dv, scale, causal, window, dtype,
                     kv_capacity, kv_ring, workspace, workspace_bytes, stream, b);
}

int sdpa_device_status(sdpa_stream_t stream, int* detail) {
  DeviceState* st = nullptr;
  if (detail) *detail = 0;
  int rc = device_state(&st);
  if (rc) return rc;
  auto strm = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(strm) != cudaSuccess) return SDPA_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (code) {
    const int zero = 0;
    if (cudaMemcpy(st->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return SDPA_ERR_CUDA;
  }
  if (detail) *detail = code;
  return code ? SDPA_ERR_DEVICE_TIMEOUT : SDPA_OK;
}

const char* sdpa_status_string(int status) {
  switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID_ARG: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported head dim or dtype";
    case SDPA_ERR_WORKSPACE: return "workspace missing or too small";
    case SDPA_ERR_CUDA: return "CUDA runtime or driver call failed";
    case SDPA_ERR_DEVICE_TIMEOUT: return "a kernel wait gave up (device timeout) or a kernel check failed";
    case SDPA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SDPA_ERR_SCRATCH_LIMIT:
      return "call needs more than the built-in scratch of sdpa_decode_noalloc";
    default: return "unknown status";
  }
}

int sdpa_version(void) { return 100; }

int sdpa_selftest_timeout(const void* q, const void* k, const void* v, void* out, int D,
                          int decode, void* workspace, size_t workspace_bytes,
                          sdpa_stream_t stream, int* detail) {
  if (detail) *detail = 0;
  if (!q || !k || !v || !out || (D != 256 && D != 512)) return SDPA_ERR_INVALID_ARG;
  if (decode == 2) {
    // Persistent prefill whose suffix pieces never publish their flags: the
    // prefix units' bounded waits run out and their tiles are stored as NaN.
    const int B = 1, Hq = 2, Hkv = 1, Lq = 256, Lk = 4096;
    if (D != 256) return SDPA_ERR_INVALID_ARG;
    int rc = validate(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, 1.f / 16.f, 1, 0, SDPA_F16);
    if (rc) return rc;
    DeviceState* st = nullptr;
    rc = device_state(&st);
    if (rc) return rc;
    const int mode = choose_mode(false, D, 0);
    const long long u = persistent_units<false>(st, mode, D, B, Hq, Hkv, Lq, Lk, 1, 0);
    if (u <= 0) return SDPA_ERR_UNSUPPORTED;
    const QTiling qt = qtiling(mode, Hq / Hkv);
    if (plan_tail(u, B, Hq, Lq, Lk, 1, 0, key_tile(mode), qt.rows, qt.heads).US <= 0)
      return SDPA_ERR_UNSUPPORTED;  // no suffix pieces on this device: nothing to withhold
    if (!workspace || workspace_bytes < sk_layout(u).bytes || !aligned16(workspace))
      return SDPA_ERR_WORKSPACE;
    rc = run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, 1.f / 16.f, 1, 0, false, 1, false,
                    workspace, reinterpret_cast<cudaStream_t>(stream), st, /*withhold=*/2, u);
    if (rc) return rc;
    return sdpa_device_status(stream, detail);
  }
  if (decode != 0 && decode != 1) return SDPA_ERR_INVALID_ARG;
  const int B = 1, Hq = 2, Hkv = 1, Lq = decode ? 1 : 128, Lk = 128;
  int rc = validate(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, 1.f / 16.f, 1, 0, SDPA_F16);
  if (rc) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  auto strm = reinterpret_cast<cudaStream_t>(stream);
  DecodePlan pl;
  if (decode) {
    pl = plan_decode(st, B, Hq, Hkv, D, D, 0);
    const size_t need = decode_partial_bytes(pl, static_cast<long long>(B) * Hq * Lq, D);
    if (need > 0 && (!workspace || workspace_bytes < need)) return SDPA_ERR_WORKSPACE;
  }
  rc = run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, 1.f / 16.f, 1, 0, decode != 0, 1, false,
                  workspace, strm, st, /*withhold_q=*/1, 0, 0, 0, 0, BiasArg(),
                  decode ? &pl : nullptr);
  if (rc) return rc;
  return sdpa_device_status(stream, detail);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free decode: the split partials go to a scratch array that is part
// of the library image instead of a caller workspace.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SDPA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device.  The array's name is only a host-side handle; the kernels must be
// given this address.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDPA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return SDPA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return SDPA_OK;
}

}  // namespace

extern "C" int sdpa_decode_noalloc(const void* q, const void* k, const void* v, void* out, int B,
                                   int Hq, int Hkv, int Lq, int Lk, int D, float scale,
                                   int causal, int window, int dtype, sdpa_stream_t stream) {
  int rc = validate(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, dtype);
  if (rc) return rc;
  if (Lq > 8) return SDPA_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  const bool bf16 = dtype == SDPA_BF16;
  const DecodePlan pl = plan_decode(st, B, Hq, Hkv, D, D, causal ? window : 0);
  if (decode_partial_bytes(pl, static_cast<long long>(B) * Hq * Lq, D) >
      SDPA_NOALLOC_SCRATCH_BYTES)
    return SDPA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  auto strm = reinterpret_cast<cudaStream_t>(stream);
  return bf16 ? run<true>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, true, 0,
                          true, scratch, strm, st, 0, 0, 0, 0, 0, BiasArg(), &pl)
              : run<false>(q, k, v, out, B, Hq, Hkv, Lq, Lk, D, scale, causal, window, true, 0,
                           true, scratch, strm, st, 0, 0, 0, 0, 0, BiasArg(), &pl);
}
