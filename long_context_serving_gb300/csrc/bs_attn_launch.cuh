// Launchers of the attention kernels (host side), shared by the stand-alone call and
// the fused decode step.
#pragma once

#include "bs_attn_plan.cuh"

namespace bsi {

struct AttnArgs {
  bs_dims dims;
  const void *q;
  bs_kv kv;
  bs_head_cfg cfg;
  const int32_t *sel_idx;
  const int32_t *sel_cnt;
  const float *bias;  // logit bias of every block [units][max_blocks_per_unit] (ED-DMA), or null
  float *out;
  float *lse;
  int32_t *arrivals;  // per-unit arrival tickets of the splits (workspace mode)
  float *records;     // split records (workspace mode)
  const int32_t *plist;  // fused step: page lists of non-streaming units, else null
  const int32_t *pub;    // fused step: published selections, (epoch << 16) | count, per unit
  int32_t *expect;       // fused step: epoch of the last selection the attention took, per unit
  int32_t *st;
  uint64_t wait_ns;      // limit of every device-side wait
};

// step = true: launched as a programmatic dependent of the fused step's selection
// kernel (streaming units run ahead, the rest wait for their unit's selection).
bs_status launch_attn_bf16(const AttnArgs &a, bool step, cudaStream_t cs);
bs_status launch_attn_f32(const AttnArgs &a, bool step, cudaStream_t cs);

// About two CTAs per SM of the current device (the attention's split target).
inline int attn_target_ctas() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2 * 148;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
    cached[dev] = 2 * sms;
  }
  return cached[dev];
}

// cudaLaunchKernelEx with an optional cluster width and programmatic serialization.
template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, dim3 grid, int threads, size_t smem, cudaStream_t cs, int cluster_x, bool pdl,
                      Args... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(threads);
  lc.dynamicSmemBytes = smem;
  lc.stream = cs;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  lc.attrs = attr;
  lc.numAttrs = n;
  return cudaLaunchKernelEx(&lc, kernel, args...);
}

}  // namespace bsi
