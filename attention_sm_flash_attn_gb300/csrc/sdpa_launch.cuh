// sdpa_launch.cuh -- per-device launch state and the launch of one attention
// kernel instantiation, shared by the translation units that instantiate them:
// sdpa_api.cu (kernels without a bias) and sdpa_bias.cu (kernels that add an
// additive bias to the scores).  Splitting the instantiations over two units
// lets them compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>

#include "sdpa_gb300.h"
#include "sdpa_kernels.cuh"

namespace gbsdpa_host {

using gbsdpa::AttnParams;
using gbsdpa::Cfg;

// Slot of a kernel instantiation in the per-device tables: bias x dtype x
// variant (6) x per-CTA head dims (Q/K, V): (256, 256), (128, 128), (192, 192),
// (192, 256).
template <bool BF16, int MODE, int HD, int HDV, bool BIAS>
constexpr int variant_index() {
  return (BIAS ? 2 * 4 * gbsdpa::kNumModes : 0) + (BF16 ? 1 : 0) +
         2 * (MODE * 4 + (HD != HDV ? 3 : HD == 256 ? 0 : HD == 128 ? 1 : 2));
}
constexpr int kNumVariants = 2 * 2 * gbsdpa::kNumModes * 4;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;                // device address of the status word
  bool attr_set[kNumVariants] = {};     // per kernel instantiation (variant_index)
  int sk_units[kNumVariants] = {};      // resident persistent units per instantiation
  // kDecode: clusters of 2^k CTAs (k = 0..4) that can be resident at once, per
  // instantiation (-1: not queried yet).
  int dec_fit[kNumVariants][5];
  unsigned long long epoch = 0;         // last persistent-launch epoch handed out
  DeviceState() {
    for (auto& row : dec_fit)
      for (int& x : row) x = -1;
  }
};

static_assert(variant_index<false, gbsdpa::kSingle, 192, 256, false>() !=
                      variant_index<false, gbsdpa::kSingle, 192, 192, false>() &&
                  variant_index<true, gbsdpa::kPairXD, 192, 256, false>() <
                      variant_index<false, gbsdpa::kSingle, 256, 256, true>() &&
                  variant_index<true, gbsdpa::kPairXD, 192, 256, true>() < kNumVariants,
              "distinct slots within the tables");

template <bool BF16, int MODE, int HD, int HDV, bool BIAS>
int ensure_attr(DeviceState* st) {
  constexpr int idx = variant_index<BF16, MODE, HD, HDV, BIAS>();
  if (st->attr_set[idx]) return SDPA_OK;
  auto kern = gbsdpa::attn_fwd_kernel<BF16, MODE, HD, HDV, BIAS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<BF16, MODE, HD, HDV, BIAS>::SMEM_BYTES) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (MODE == gbsdpa::kDecode &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return SDPA_ERR_CUDA;
  st->attr_set[idx] = true;
  return SDPA_OK;
}

// CTAs per cluster of a launch: 2 for the pair variants, the planned decode
// cluster for kDecode, none (1) for kSingle.
template <int MODE>
int cluster_ctas(const AttnParams& p) {
  if (MODE == gbsdpa::kSingle) return 1;
  if (MODE == gbsdpa::kDecode) return p.dec_cs;
  return 2;
}

template <bool BF16, int MODE, int HD, int HDV, bool BIAS>
void fill_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, long long ctas, int cluster,
                 cudaStream_t stream) {
  *cfg = {};
  cfg->gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg->blockDim = dim3(Cfg<BF16, MODE, HD, HDV, BIAS>::NTHREADS, 1, 1);
  cfg->dynamicSmemBytes = Cfg<BF16, MODE, HD, HDV, BIAS>::SMEM_BYTES;
  cfg->stream = stream;
  cfg->attrs = attr;
  cfg->numAttrs = 0;
  if (cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->numAttrs = 1;
  }
}

template <bool BF16, int MODE, int HD, int HDV, bool BIAS>
int launch_attn(const AttnParams& p, long long items, cudaStream_t stream, DeviceState* st) {
  int rc = ensure_attr<BF16, MODE, HD, HDV, BIAS>(st);
  if (rc) return rc;
  // items: CTA pairs of the pair variants, CTAs otherwise (decode clusters
  // are groups of consecutive items).
  const int cl = cluster_ctas<MODE>(p);
  const long long ctas = items * (MODE == gbsdpa::kDecode ? 1 : cl);
  if (ctas <= 0 || ctas > 0x7fffffffll || cl < 1 || ctas % cl != 0) return SDPA_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  // A persistent grid waits on itself (prefix units on suffix units).  It is
  // sized to the occupancy limit, so on an otherwise idle GPU all of it is
  // resident; the kernel starts the never-waiting units first, and a wait that
  // still runs out reports a device timeout instead of hanging.
  fill_launch<BF16, MODE, HD, HDV, BIAS>(&cfg, attr, ctas, cl, stream);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, gbsdpa::attn_fwd_kernel<BF16, MODE, HD, HDV, BIAS>, p);
  return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA;
}

// How many persistent units (CTAs, or CTA pairs for the 2-SM variant) can be
// resident at once on this device; 0 if the variant cannot run persistently.
template <bool BF16, int MODE, int HD, int HDV, bool BIAS>
int resident_units(DeviceState* st) {
  constexpr int idx = variant_index<BF16, MODE, HD, HDV, BIAS>();
  if (st->sk_units[idx]) return st->sk_units[idx];
  if (ensure_attr<BF16, MODE, HD, HDV, BIAS>(st)) return 0;
  auto kern = gbsdpa::attn_fwd_kernel<BF16, MODE, HD, HDV, BIAS>;
  int units = 0;
  if (MODE == gbsdpa::kSingle) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern,
                                                      Cfg<BF16, MODE, HD, HDV, BIAS>::NTHREADS,
                                                      Cfg<BF16, MODE, HD, HDV, BIAS>::SMEM_BYTES) !=
        cudaSuccess)
      return 0;
    units = per_sm * st->sms;
  } else {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch<BF16, MODE, HD, HDV, BIAS>(&cfg, attr, 2 * (st->sms / 2), 2, nullptr);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) return 0;
    units = clusters;
  }
  st->sk_units[idx] = std::max(0, units);
  return st->sk_units[idx];
}

// kDecode: how many clusters of `cs` CTAs (a power of two up to 16) can be
// resident at once (0: such clusters cannot launch).
template <bool BF16, int HD, int HDV>
int decode_clusters_fit(DeviceState* st, int cs) {
  constexpr int idx = variant_index<BF16, gbsdpa::kDecode, HD, HDV, false>();
  int k = 0;
  while ((1 << k) < cs) ++k;
  if (k > 4 || (1 << k) != cs) return 0;
  if (st->dec_fit[idx][k] >= 0) return st->dec_fit[idx][k];
  if (ensure_attr<BF16, gbsdpa::kDecode, HD, HDV, false>(st)) return 0;
  auto kern = gbsdpa::attn_fwd_kernel<BF16, gbsdpa::kDecode, HD, HDV, false>;
  int fit = 0;
  if (cs == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, kern, Cfg<BF16, gbsdpa::kDecode, HD, HDV, false>::NTHREADS,
            Cfg<BF16, gbsdpa::kDecode, HD, HDV, false>::SMEM_BYTES) == cudaSuccess)
      fit = per_sm * st->sms;
  } else {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch<BF16, gbsdpa::kDecode, HD, HDV, false>(&cfg, attr, cs * (st->sms / cs), cs,
                                                       nullptr);
    if (cudaOccupancyMaxActiveClusters(&fit, kern, &cfg) != cudaSuccess) fit = 0;
  }
  st->dec_fit[idx][k] = fit > 0 ? fit : 0;
  return st->dec_fit[idx][k];
}

// kDecode clusters of `cs` CTAs resident at once for these head dims (fp16 and
// bf16 instantiations have the same footprint).
inline int decode_fit(int D, int Dv, DeviceState* st, int cs) {
  return D != Dv    ? decode_clusters_fit<false, 192, 256>(st, cs)
         : D == 128 ? decode_clusters_fit<false, 128, 128>(st, cs)
         : D == 192 ? decode_clusters_fit<false, 192, 192>(st, cs)
                    : decode_clusters_fit<false, 256, 256>(st, cs);
}

// Run-time choice of the instantiation: variant `mode`, Q/K head dim D, V head
// dim Dv (the pairs the host validation admits).
template <bool BF16, bool BIAS>
int launch_variant(int mode, int D, int Dv, const AttnParams& p, long long items,
                   cudaStream_t stream, DeviceState* st) {
  using gbsdpa::kDuo;
  using gbsdpa::kDuoQ;
  using gbsdpa::kSingle;
  switch (mode) {
    case gbsdpa::kPairX: return launch_attn<BF16, gbsdpa::kPairX, 256, 256, BIAS>(p, items, stream, st);
    case gbsdpa::kPairXD:
      return launch_attn<BF16, gbsdpa::kPairXD, 256, 256, BIAS>(p, items, stream, st);
    case kDuoQ:
      if constexpr (!BIAS)
        return launch_attn<BF16, kDuoQ, 256, 256, false>(p, items, stream, st);
      else
        return SDPA_ERR_INVALID_ARG;  // never chosen with a bias
    case kDuo:
      return D == 128 ? launch_attn<BF16, kDuo, 128, 128, BIAS>(p, items, stream, st)
                      : launch_attn<BF16, kDuo, 256, 256, BIAS>(p, items, stream, st);
    case gbsdpa::kDecode:
      return D != Dv    ? launch_attn<BF16, gbsdpa::kDecode, 192, 256, BIAS>(p, items, stream, st)
             : D == 128 ? launch_attn<BF16, gbsdpa::kDecode, 128, 128, BIAS>(p, items, stream, st)
             : D == 192 ? launch_attn<BF16, gbsdpa::kDecode, 192, 192, BIAS>(p, items, stream, st)
                        : launch_attn<BF16, gbsdpa::kDecode, 256, 256, BIAS>(p, items, stream, st);
    default:
      return D != Dv    ? launch_attn<BF16, kSingle, 192, 256, BIAS>(p, items, stream, st)
             : D == 128 ? launch_attn<BF16, kSingle, 128, 128, BIAS>(p, items, stream, st)
             : D == 192 ? launch_attn<BF16, kSingle, 192, 192, BIAS>(p, items, stream, st)
                        : launch_attn<BF16, kSingle, 256, 256, BIAS>(p, items, stream, st);
  }
}

// Resident persistent units of the instantiation a prefill with these head dims
// runs (0: not persistent: the head-dim-split pair, or a failed query).
template <bool BF16, bool BIAS>
int resident_variant(int mode, int D, int Dv, DeviceState* st) {
  using gbsdpa::kDuo;
  using gbsdpa::kDuoQ;
  using gbsdpa::kSingle;
  if (mode == kDuoQ) {
    if constexpr (!BIAS)
      return resident_units<BF16, kDuoQ, 256, 256, false>(st);
    else
      return 0;
  }
  if (mode == kSingle)
    return D != Dv    ? resident_units<BF16, kSingle, 192, 256, BIAS>(st)
           : D == 128 ? resident_units<BF16, kSingle, 128, 128, BIAS>(st)
           : D == 192 ? resident_units<BF16, kSingle, 192, 192, BIAS>(st)
                      : resident_units<BF16, kSingle, 256, 256, BIAS>(st);
  if (mode == kDuo)
    return D == 128 ? resident_units<BF16, kDuo, 128, 128, BIAS>(st)
                    : resident_units<BF16, kDuo, 256, 256, BIAS>(st);
  return 0;
}

// The kernels with a bias, instantiated in sdpa_bias.cu.
int launch_bias_variant(bool bf16, int mode, int D, int Dv, const AttnParams& p, long long items,
                        cudaStream_t stream, DeviceState* st);
int resident_bias_variant(bool bf16, int mode, int D, int Dv, DeviceState* st);

}  // namespace gbsdpa_host
