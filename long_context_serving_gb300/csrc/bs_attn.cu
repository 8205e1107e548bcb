// a4: sparse decode attention over the selected blocks ("Technische Samenvatting:
// Fluxion", Probleemstelling item 1: top-k selection, then sparse attention over the
// selected KV blocks; Kerninzichten item 3: this work is bound by data movement).
//
// Split-KV flash-decode. A unit's selected blocks cover n_pages pages of 16 tokens;
// they are cut into at most 32 splits of pps pages (pps a multiple of 4, chosen from
// n_pages alone). One CTA of 256 threads per (split, unit):
//   * warp 0 resolves the page table and issues one 1-D bulk copy (TMA) per K page
//     and per V page into a two-deep ring of 4-page stages, each signalling an
//     mbarrier with its byte count;
//   * q.K: four threads per token, each over every fourth 16-byte chunk of the row
//     in a token-rotated order (conflict-free shared-memory phases), q in shared
//     memory pre-scaled by log2(e)/sqrt(d); a two-step xor shuffle completes the dot;
//   * online softmax per head (one warp per head, base-2 exponent, fp32);
//   * P.V: warp w takes tokens w, w+8, ...; lane l owns head_dim/32 dimensions and
//     accumulates all G heads;
//   * the 8 warps' accumulators are summed through shared memory and the split writes
//     its (o, m, l) record to the workspace;
//   * the last split of a unit to finish (an integer arrival ticket per unit) merges
//     the unit's records in split order by log-sum-exp and writes out and lse. A unit
//     with a single split writes its output directly.
// Tokens past T inside a partial tail page are masked out of both products.
#include <math.h>

#include "bs_attn_plan.cuh"
#include "bs_internal.cuh"

namespace bsi {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename KT>
struct KvTraits;
template <>
struct KvTraits<uint16_t> {
  static constexpr int kElemsPerChunk = 8;  // bf16 per 16 bytes
};
template <>
struct KvTraits<float> {
  static constexpr int kElemsPerChunk = 4;
};

// 16-byte chunk of K (as raw words) -> floats.
template <typename KT>
__device__ __forceinline__ void widen_chunk(const uint4 &w, float (&k)[KvTraits<KT>::kElemsPerChunk]);
template <>
__device__ __forceinline__ void widen_chunk<uint16_t>(const uint4 &w, float (&k)[8]) {
  k[0] = bf16lo(w.x); k[1] = bf16hi(w.x); k[2] = bf16lo(w.y); k[3] = bf16hi(w.y);
  k[4] = bf16lo(w.z); k[5] = bf16hi(w.z); k[6] = bf16lo(w.w); k[7] = bf16hi(w.w);
}
template <>
__device__ __forceinline__ void widen_chunk<float>(const uint4 &w, float (&k)[4]) {
  k[0] = __uint_as_float(w.x); k[1] = __uint_as_float(w.y);
  k[2] = __uint_as_float(w.z); k[3] = __uint_as_float(w.w);
}

// head_dim/32 values of a V row owned by one lane -> floats.
template <int DPL, typename KT>
__device__ __forceinline__ void load_v(const KT *p, float (&v)[DPL]);
template <>
__device__ __forceinline__ void load_v<4, uint16_t>(const uint16_t *p, float (&v)[4]) {
  const uint2 w = *reinterpret_cast<const uint2 *>(p);
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
}
template <>
__device__ __forceinline__ void load_v<2, uint16_t>(const uint16_t *p, float (&v)[2]) {
  const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
  v[0] = bf16lo(w); v[1] = bf16hi(w);
}
template <>
__device__ __forceinline__ void load_v<4, float>(const float *p, float (&v)[4]) {
  const float4 w = *reinterpret_cast<const float4 *>(p);
  v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
}
template <>
__device__ __forceinline__ void load_v<2, float>(const float *p, float (&v)[2]) {
  const float2 w = *reinterpret_cast<const float2 *>(p);
  v[0] = w.x; v[1] = w.y;
}

template <int D, typename KT, int G>
struct AttnLayout {
  static constexpr int kPageBytes = kPage * D * static_cast<int>(sizeof(KT));
  static constexpr int kStageBytes = kStagePages * kPageBytes;
  static constexpr int kGP = (G + 3) & ~3;  // p row stride (floats)
  static constexpr int kOffQ = 4 * kStageBytes;
  static constexpr int kOffS = kOffQ + G * D * 4;
  static constexpr int kOffP = kOffS + G * kStageTokens * 4;
  static constexpr int kOffA = kOffP + kStageTokens * kGP * 4;
  static constexpr int kBytes = kOffA + kMaxG * 4;
  static_assert(2 * kStageBytes >= 8 * G * D * 4, "reduction scratch must fit in the K stages");
};

// Validated per-unit view: selection size, gathered pages and split plan.
struct UnitView {
  bool ok;
  int T, g, cnt;
  UnitPages pg;
};

__device__ __forceinline__ UnitView unit_view(const bs_dims &dims, const bs_kv &kv, const bs_head_cfg &cfg,
                                              const int32_t *sel_idx, const int32_t *sel_cnt, int u,
                                              int32_t *st, bool may_report) {
  UnitView v;
  v.ok = false;
  const int b = u / dims.n_kv_heads;
  v.T = kv.seq_lens[b];
  v.g = cfg.block_tokens[u];
  v.cnt = sel_cnt[u];
  v.pg.n_pages = 0;
  v.pg.n_split = 0;
  if (v.g <= 0 || v.g % kPage != 0 || v.T < 1 || v.cnt < 0 || v.cnt > dims.max_sel_per_unit) {
    if (may_report) report(st, BS_ERR_INVALID_ARG);
    return v;
  }
  if (v.cnt == 0) return v;
  const int last = sel_idx[static_cast<size_t>(u) * dims.max_sel_per_unit + v.cnt - 1];
  if (last < 0 || static_cast<int64_t>(last) * v.g >= v.T) {
    if (may_report) report(st, BS_ERR_DEVICE_BOUNDS);
    return v;
  }
  v.pg = unit_pages(v.T, v.g, v.cnt, last);
  v.ok = v.pg.n_pages > 0;
  return v;
}

template <int D, typename KT, int G>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(bs_dims dims, const void *__restrict__ q,
                                                                  bs_kv kv, bs_head_cfg cfg,
                                                                  const int32_t *__restrict__ sel_idx,
                                                                  const int32_t *__restrict__ sel_cnt,
                                                                  int32_t *__restrict__ arrivals,
                                                                  float *__restrict__ ws, float *__restrict__ out,
                                                                  float *__restrict__ lse, int32_t *st) {
  using L = AttnLayout<D, KT, G>;
  constexpr int DPL = D / 32;
  constexpr int EPC = KvTraits<KT>::kElemsPerChunk;
  constexpr int kChunks = D * static_cast<int>(sizeof(KT)) / 16;  // 16-byte chunks per row
  constexpr int kPer = kChunks / 4;                                // per quarter (power of two)
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bars[2];
  __shared__ int slot_valid[2][kStagePages];

  const int u = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const UnitView uv = unit_view(dims, kv, cfg, sel_idx, sel_cnt, u, st, split == 0 && tid == 0);
  const int b = u / dims.n_kv_heads, hk = u % dims.n_kv_heads;
  constexpr int QD = D / 4;
  const size_t orow0 = static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G;
  if (!uv.ok) {
    // Nothing to attend (or an invalid unit): zero output, lse = -inf.
    if (split == 0)
      for (int i = tid; i < G * QD; i += kAttnThreads) {
        reinterpret_cast<float4 *>(out + (orow0 + i / QD) * D)[i % QD] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i % QD == 0) lse[orow0 + i / QD] = -INFINITY;
      }
    return;
  }
  if (split >= uv.pg.n_split) return;
  const int ppb = uv.pg.ppb;
  const int gp0 = split * uv.pg.pps;
  const int gp1 = min(gp0 + uv.pg.pps, uv.pg.n_pages);
  const int n_stages = (gp1 - gp0 + kStagePages - 1) / kStagePages;
  const int32_t *sel = sel_idx + static_cast<size_t>(u) * dims.max_sel_per_unit;
  const int32_t *pt = kv.page_table + static_cast<size_t>(u) * dims.max_pages_per_unit;
  const unsigned char *kpool = static_cast<const unsigned char *>(kv.k_pool);
  const unsigned char *vpool = static_cast<const unsigned char *>(kv.v_pool);

  float *qs = reinterpret_cast<float *>(smem + L::kOffQ);
  float *s_sm = reinterpret_cast<float *>(smem + L::kOffS);
  float *p_sm = reinterpret_cast<float *>(smem + L::kOffP);
  float *alpha_sm = reinterpret_cast<float *>(smem + L::kOffA);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Warp 0: resolve the 4 pages of a stage and start their copies.
  auto issue = [&](int stage, int buf) {
    int valid_tok = 0, phys = -1;
    const int gp = gp0 + stage * kStagePages + lane;
    if (lane < kStagePages && gp < gp1) {
      const int i = gp / ppb, pb = gp - (gp / ppb) * ppb;
      const int c = sel[i];
      const int lp = c * ppb + pb;
      const int t0 = lp * kPage;
      if (c < 0 || lp >= dims.max_pages_per_unit || t0 >= uv.T) {
        report(st, BS_ERR_DEVICE_BOUNDS);
      } else {
        phys = __ldg(pt + lp);
        if (phys < 0 || phys >= dims.n_pages) report(st, BS_ERR_DEVICE_BOUNDS);
        else valid_tok = min(kPage, uv.T - t0);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, valid_tok > 0);
    if (lane == 0) mbar_arrive_expect_tx(&bars[buf], static_cast<uint32_t>(__popc(m)) * 2u * L::kPageBytes);
    __syncwarp();
    if (valid_tok > 0) {
      fence_proxy_async_smem();
      const size_t src = static_cast<size_t>(phys) * L::kPageBytes;
      bulk_g2s(smem + buf * L::kStageBytes + lane * L::kPageBytes, kpool + src, L::kPageBytes, &bars[buf]);
      bulk_g2s(smem + (2 + buf) * L::kStageBytes + lane * L::kPageBytes, vpool + src, L::kPageBytes, &bars[buf]);
    }
    if (lane < kStagePages) slot_valid[buf][lane] = valid_tok;
  };

  if (warp == 0) {
    issue(0, 0);
    if (n_stages > 1) issue(1, 1);
  }
  {
    const float qscale = rsqrtf(static_cast<float>(D)) * kLog2e;
    const size_t qbase = (static_cast<size_t>(b) * dims.n_q_heads + static_cast<size_t>(hk) * G) * D;
    for (int i = tid; i < G * D; i += kAttnThreads) qs[i] = load_scalar(q, qbase + i, dims.q_dtype) * qscale;
  }

  float m_run = -INFINITY, l_run = 0.0f;  // per head, kept by warp h (lane-replicated)
  float acc[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[h][j] = 0.0f;

  const int tok = tid >> 2, qq = tid & 3;
  for (int it = 0; it < n_stages; ++it) {
    const int buf = it & 1;
    const bool ok = mbar_wait_bounded(&bars[buf], static_cast<uint32_t>((it >> 1) & 1), st);
    if (__syncthreads_or(!ok)) return;

    // ---- scores s = q.k (log2 units) --------------------------------------
    const unsigned char *Kb = smem + buf * L::kStageBytes;
    const bool tvalid = (tok & (kPage - 1)) < slot_valid[buf][tok >> 4];
    float a[G];
#pragma unroll
    for (int h = 0; h < G; ++h) a[h] = 0.0f;
    if (tvalid) {
      const uint4 *row = reinterpret_cast<const uint4 *>(Kb + tok * D * sizeof(KT));
#pragma unroll
      for (int c = 0; c < kPer; ++c) {
        const int ch = qq + 4 * ((c + tok) & (kPer - 1));
        float kf[EPC];
        widen_chunk<KT>(row[ch], kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 *qv = reinterpret_cast<const float4 *>(qs + h * D + ch * EPC);
#pragma unroll
          for (int e4 = 0; e4 < EPC / 4; ++e4) {
            const float4 q4 = qv[e4];
            a[h] = fmaf(q4.x, kf[4 * e4 + 0], a[h]);
            a[h] = fmaf(q4.y, kf[4 * e4 + 1], a[h]);
            a[h] = fmaf(q4.z, kf[4 * e4 + 2], a[h]);
            a[h] = fmaf(q4.w, kf[4 * e4 + 3], a[h]);
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 1);
      a[h] += __shfl_xor_sync(0xffffffffu, a[h], 2);
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
      if ((h & 3) == qq) s_sm[h * kStageTokens + tok] = tvalid ? a[h] : -INFINITY;
    __syncthreads();

    // ---- online softmax, one warp per head ---------------------------------
    if (warp < G) {
      const float s0 = s_sm[warp * kStageTokens + lane];
      const float s1 = s_sm[warp * kStageTokens + lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run, mx);
      float alpha = 1.0f, p0 = 0.0f, p1 = 0.0f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_run - m_new);
        p0 = exp2f(s0 - m_new);
        p1 = exp2f(s1 - m_new);
      }
      float ps = p0 + p1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l_run = l_run * alpha + ps;
      m_run = m_new;
      p_sm[lane * L::kGP + warp] = p0;
      p_sm[(lane + 32) * L::kGP + warp] = p1;
      if (lane == 0) alpha_sm[warp] = alpha;
    }
    __syncthreads();

    // ---- o += p V ------------------------------------------------------------
    {
      float al[G];
#pragma unroll
      for (int h = 0; h < G; ++h) al[h] = alpha_sm[h];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] *= al[h];
      const KT *Vb = reinterpret_cast<const KT *>(smem + (2 + buf) * L::kStageBytes);
#pragma unroll 2
      for (int i = 0; i < kStageTokens / 8; ++i) {
        const int t = warp + 8 * i;
        if ((t & (kPage - 1)) >= slot_valid[buf][t >> 4]) continue;  // warp-uniform
        float v[DPL];
        load_v<DPL, KT>(Vb + t * D + lane * DPL, v);
        float p[L::kGP];
#pragma unroll
        for (int h4 = 0; h4 < L::kGP / 4; ++h4) {
          const float4 pv = reinterpret_cast<const float4 *>(p_sm + t * L::kGP)[h4];
          p[4 * h4 + 0] = pv.x; p[4 * h4 + 1] = pv.y; p[4 * h4 + 2] = pv.z; p[4 * h4 + 3] = pv.w;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int j = 0; j < DPL; ++j) acc[h][j] = fmaf(p[h], v[j], acc[h][j]);
      }
    }
    __syncthreads();
    if (warp == 0 && it + 2 < n_stages) issue(it + 2, buf);
  }

  // ---- sum the 8 warps' accumulators ------------------------------------------
  float *red = reinterpret_cast<float *>(smem);  // [8][G][D] over the K stages
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) red[(warp * G + h) * D + lane * DPL + j] = acc[h][j];
  __shared__ float ml_sm[2][kMaxG];
  if (warp < G && lane == 0) {
    ml_sm[0][warp] = m_run;
    ml_sm[1][warp] = l_run;
  }
  __syncthreads();
  constexpr int REC = attn_record_floats(D);
  if (uv.pg.n_split == 1) {
    // Single split: normalise and write the output directly.
    for (int i = tid; i < G * QD; i += kAttnThreads) {
      const int h = i / QD, dq = i % QD;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 r = reinterpret_cast<const float4 *>(red + (w * G + h) * D)[dq];
        o.x += r.x; o.y += r.y; o.z += r.z; o.w += r.w;
      }
      const float inv = 1.0f / ml_sm[1][h];
      o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
      reinterpret_cast<float4 *>(out + (orow0 + h) * D)[dq] = o;
      if (dq == 0) lse[orow0 + h] = (ml_sm[0][h] + log2f(ml_sm[1][h])) * kLn2;
    }
    return;
  }
  float *rec = ws + (static_cast<size_t>(u) * kAttnMaxSplits + split) * G * REC;
  for (int i = tid; i < G * QD; i += kAttnThreads) {
    const int h = i / QD, dq = i % QD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float4 r = reinterpret_cast<const float4 *>(red + (w * G + h) * D)[dq];
      o.x += r.x; o.y += r.y; o.z += r.z; o.w += r.w;
    }
    reinterpret_cast<float4 *>(rec + h * REC)[dq] = o;
  }
  if (tid < G) {
    rec[tid * REC + D] = ml_sm[0][tid];
    rec[tid * REC + D + 1] = ml_sm[1][tid];
  }
  // Publish the record, then take an arrival ticket; the last split merges.
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (tid == 0) is_last = (atomicAdd(arrivals + u, 1) == uv.pg.n_split - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // Merge: M = max m_i, L = sum l_i 2^(m_i - M), o = sum 2^(m_i - M) o_i / L,
  // lse = ln 2 (M + log2 L); splits are visited in index order.
  const float *base = ws + static_cast<size_t>(u) * kAttnMaxSplits * G * REC;
  for (int i = tid; i < G * QD; i += kAttnThreads) {
    const int h = i / QD, dq = i % QD;
    const float *hb = base + h * REC;
    float M = -INFINITY;
    for (int sp = 0; sp < uv.pg.n_split; ++sp) M = fmaxf(M, __ldcg(hb + static_cast<size_t>(sp) * G * REC + D));
    float Lsum = 0.0f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < uv.pg.n_split; ++sp) {
      const float *r = hb + static_cast<size_t>(sp) * G * REC;
      const float mi = __ldcg(r + D);
      const float w = (mi == -INFINITY) ? 0.0f : exp2f(mi - M);
      Lsum = fmaf(__ldcg(r + D + 1), w, Lsum);
      const float4 oi = __ldcg(reinterpret_cast<const float4 *>(r) + dq);
      o.x = fmaf(oi.x, w, o.x);
      o.y = fmaf(oi.y, w, o.y);
      o.z = fmaf(oi.z, w, o.z);
      o.w = fmaf(oi.w, w, o.w);
    }
    const float inv = 1.0f / Lsum;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
    reinterpret_cast<float4 *>(out + (orow0 + h) * D)[dq] = o;
    if (dq == 0) lse[orow0 + h] = (M + log2f(Lsum)) * kLn2;
  }
  if (tid == 0) arrivals[u] = 0;  // ready for the next call
}

template <int D, typename KT, int G>
bs_status launch_attn(const bs_dims &dims, const void *q, const bs_kv &kv, const bs_head_cfg &cfg,
                      const int32_t *sel_idx, const int32_t *sel_cnt, float *out, float *lse, float *ws,
                      int32_t *st, cudaStream_t cs) {
  using L = AttnLayout<D, KT, G>;
  static const cudaError_t attr = cudaFuncSetAttribute(attn_split_kernel<D, KT, G>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (attr != cudaSuccess) return BS_ERR_CUDA;
  const int units = dims.batch * dims.n_kv_heads;
  int splits = (dims.max_gather_pages_per_unit + kStagePages - 1) / kStagePages;
  if (splits > kAttnMaxSplits) splits = kAttnMaxSplits;
  if (splits < 1) splits = 1;
  int32_t *arrivals = reinterpret_cast<int32_t *>(ws);
  float *records = ws + attn_counter_floats(units);
  attn_split_kernel<D, KT, G><<<dim3(splits, units), kAttnThreads, L::kBytes, cs>>>(
      dims, q, kv, cfg, sel_idx, sel_cnt, arrivals, records, out, lse, st);
  return launch_status();
}

template <int D, typename KT>
bs_status dispatch_g(int G, const bs_dims &dims, const void *q, const bs_kv &kv, const bs_head_cfg &cfg,
                     const int32_t *sel_idx, const int32_t *sel_cnt, float *out, float *lse, float *ws,
                     int32_t *st, cudaStream_t cs) {
  switch (G) {
    case 1: return launch_attn<D, KT, 1>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 2: return launch_attn<D, KT, 2>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 3: return launch_attn<D, KT, 3>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 4: return launch_attn<D, KT, 4>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 5: return launch_attn<D, KT, 5>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 6: return launch_attn<D, KT, 6>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    case 7: return launch_attn<D, KT, 7>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
    default: return launch_attn<D, KT, 8>(dims, q, kv, cfg, sel_idx, sel_cnt, out, lse, ws, st, cs);
  }
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_sparse_decode_attn(const bs_dims *dims, const void *q, const bs_kv *kv,
                                           const bs_head_cfg *cfg, const int32_t *sel_idx, const int32_t *sel_cnt,
                                           float *out, float *lse, void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !kv || !cfg || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens || !cfg->block_tokens ||
      !sel_idx || !sel_cnt || !out || !lse || !workspace || !dev_status)
    return BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(out) ||
      !aligned16(workspace))
    return BS_ERR_ALIGN;
  if (workspace_bytes < bs_workspace_size(dims)) return BS_ERR_CAPACITY;
  const int G = dims->n_q_heads / dims->n_kv_heads;
  float *ws = static_cast<float *>(workspace);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dims->head_dim == 128) {
    if (dims->kv_dtype == BS_BF16)
      return dispatch_g<128, uint16_t>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
    return dispatch_g<128, float>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  }
  if (dims->kv_dtype == BS_BF16)
    return dispatch_g<64, uint16_t>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  return dispatch_g<64, float>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
}

// ---------------------------------------------------------------------------
// Attention without a caller-provided workspace.
//
// Some callers cannot hand this library a workspace: a plugin running inside a host
// engine that owns every device allocation and exposes no allocator, or a serving
// loop that forbids cudaMalloc after start-up because it synchronises the device and
// can fail under memory pressure. For them the split records and arrival counters
// live in a fixed array in this library's own device memory. Each GPU that loads the
// library holds the array until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace bsi {
namespace {

constexpr size_t kFixedScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_fixed_scratch_mu;
void *g_fixed_scratch_addr[kMaxDevices] = {};

// Device address of g_fixed_scratch on the current device. In host code the array's
// name only stands in for the symbol; the address is looked up once per device (with
// that device current) and cached.
bs_status fixed_scratch_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  if (g_fixed_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fixed_scratch) != cudaSuccess || p == nullptr) return BS_ERR_CUDA;
    g_fixed_scratch_addr[dev] = p;
  }
  *addr = g_fixed_scratch_addr[dev];
  return BS_OK;
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_sparse_decode_attn_noalloc(const bs_dims *dims, const void *q, const bs_kv *kv,
                                                   const bs_head_cfg *cfg, const int32_t *sel_idx,
                                                   const int32_t *sel_cnt, float *out, float *lse,
                                                   int32_t *dev_status, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !kv || !cfg || !kv->k_pool || !kv->v_pool || !kv->page_table || !kv->seq_lens || !cfg->block_tokens ||
      !sel_idx || !sel_cnt || !out || !lse || !dev_status)
    return BS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv->k_pool) || !aligned16(kv->v_pool) || !aligned16(out)) return BS_ERR_ALIGN;
  const size_t need = bs_workspace_size(dims);
  if (need > kFixedScratchBytes) return BS_ERR_CAPACITY;
  void *scratch = nullptr;
  s = fixed_scratch_address(&scratch);
  if (s != BS_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // The arrival counters must start at zero; the array keeps whatever the previous
  // call (possibly one that stopped early) left in it.
  const size_t units = static_cast<size_t>(dims->batch) * dims->n_kv_heads;
  if (cudaMemsetAsync(scratch, 0, attn_counter_floats(units) * sizeof(float), cs) != cudaSuccess) return BS_ERR_CUDA;
  const int G = dims->n_q_heads / dims->n_kv_heads;
  float *ws = static_cast<float *>(scratch);
  if (dims->head_dim == 128) {
    if (dims->kv_dtype == BS_BF16)
      return dispatch_g<128, uint16_t>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
    return dispatch_g<128, float>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  }
  if (dims->kv_dtype == BS_BF16)
    return dispatch_g<64, uint16_t>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
  return dispatch_g<64, float>(G, *dims, q, *kv, *cfg, sel_idx, sel_cnt, out, lse, ws, dev_status, cs);
}
