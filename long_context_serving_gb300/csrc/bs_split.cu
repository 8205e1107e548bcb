// CPU/GPU split attention with a log-sum-exp merge: "Technische Samenvatting:
// Fluxion", Kerninzichten item 3 (sparse attention is bound by data movement, so the
// CPU can serve the part of a step whose KV sits in host memory) and
// Systeemcomponenten (CPU and GPU work on one step in parallel, their partial results
// combined).
//
// bs_cpu_sparse_attn: the attention of a block subset per unit on the host cores, over
// host-resident pools and host copies of the tables (fp32 arithmetic, one pass of
// online softmax per head, units spread over std::threads). bs_lse_merge: one GPU
// thread per 4 output columns of a query head combines two partial (o, lse) results.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <thread>
#include <vector>

#include "bs_internal.cuh"

namespace bsi {
namespace {

inline float bf16_to_f32_host(uint16_t h) {
  uint32_t b = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}

inline float kv_at(const void *pool, int dtype, size_t idx) {
  return dtype == BS_BF16 ? bf16_to_f32_host(static_cast<const uint16_t *>(pool)[idx])
                          : static_cast<const float *>(pool)[idx];
}

// Attention of unit u over its listed blocks (tokens clipped to T). Returns false on
// a bad page or block index.
bool cpu_unit(const bs_dims &d, const void *q, const bs_host_tables &t, const void *k_pool, const void *v_pool,
              int64_t n_pages, const int32_t *blocks, int cnt, int u, float *out, float *lse) {
  const int D = d.head_dim, G = d.n_q_heads / d.n_kv_heads;
  const int b = u / d.n_kv_heads, hk = u % d.n_kv_heads;
  const int T = t.seq_lens[b], g = t.block_tokens[u];
  const float scale = 1.0f / sqrtf(static_cast<float>(D));
  std::vector<float> qs(static_cast<size_t>(G) * D), o(static_cast<size_t>(G) * D, 0.0f), k(D), v(D);
  std::vector<float> m(G, -INFINITY), l(G, 0.0f), s(G);
  const size_t q0 = (static_cast<size_t>(b) * d.n_q_heads + static_cast<size_t>(hk) * G) * D;
  for (int i = 0; i < G * D; ++i) qs[i] = kv_at(q, d.q_dtype, q0 + i) * scale;
  bool ok = true;
  for (int j = 0; j < cnt; ++j) {
    const int c = blocks[j];
    if (c < 0 || static_cast<int64_t>(c) * g >= T) {
      ok = false;
      continue;
    }
    // ED-DMA: the block's logit is added to each of its tokens' logits; -inf drops it.
    float eb = 0.0f;
    if (t.evict_bias != nullptr) {
      if (c >= t.max_blocks_per_unit) {
        ok = false;
        continue;
      }
      eb = t.evict_bias[static_cast<size_t>(u) * t.max_blocks_per_unit + c];
      if (eb == -INFINITY) continue;
    }
    const int t1 = std::min(T, (c + 1) * g);
    for (int tok = c * g; tok < t1; ++tok) {
      const int lp = tok / kPage;
      if (lp >= d.max_pages_per_unit) {
        ok = false;
        break;
      }
      const int phys = t.page_table[static_cast<size_t>(u) * d.max_pages_per_unit + lp];
      if (phys < 0 || phys >= n_pages) {
        ok = false;
        continue;
      }
      const size_t base = (static_cast<size_t>(phys) * kPage + tok % kPage) * D;
      for (int i = 0; i < D; ++i) {
        k[i] = kv_at(k_pool, d.kv_dtype, base + i);
        v[i] = kv_at(v_pool, d.kv_dtype, base + i);
      }
      for (int h = 0; h < G; ++h) {
        float acc = 0.0f;
        for (int i = 0; i < D; ++i) acc = fmaf(qs[h * D + i], k[i], acc);
        s[h] = acc + eb;
      }
      for (int h = 0; h < G; ++h) {
        const float mn = std::max(m[h], s[h]);
        const float a = expf(m[h] - mn), p = expf(s[h] - mn);
        l[h] = l[h] * a + p;
        for (int i = 0; i < D; ++i) o[h * D + i] = fmaf(p, v[i], o[h * D + i] * a);
        m[h] = mn;
      }
    }
  }
  for (int h = 0; h < G; ++h) {
    const size_t row = static_cast<size_t>(b) * d.n_q_heads + static_cast<size_t>(hk) * G + h;
    const bool empty = l[h] == 0.0f;
    for (int i = 0; i < D; ++i) out[row * D + i] = empty ? 0.0f : o[h * D + i] / l[h];
    lse[row] = empty ? -INFINITY : m[h] + logf(l[h]);
  }
  return ok;
}

__global__ void lse_merge_kernel(int rows, int D, const float *__restrict__ oa, const float *__restrict__ la,
                                 const float *__restrict__ ob, const float *__restrict__ lb, float *out, float *lse) {
  const int QD = D / 4;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * QD) return;
  const int r = i / QD, dq = i % QD;
  const float a = la[r], bb = lb[r];
  const float M = fmaxf(a, bb);
  const float wa = a == -INFINITY ? 0.0f : expf(a - M);
  const float wb = bb == -INFINITY ? 0.0f : expf(bb - M);
  const float L = wa + wb;
  const float4 x = reinterpret_cast<const float4 *>(oa)[i], y = reinterpret_cast<const float4 *>(ob)[i];
  float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  if (L > 0.0f) {
    const float inv = 1.0f / L;
    z.x = (wa * x.x + wb * y.x) * inv;
    z.y = (wa * x.y + wb * y.y) * inv;
    z.z = (wa * x.z + wb * y.z) * inv;
    z.w = (wa * x.w + wb * y.w) * inv;
  }
  // every thread of the row reads la / lb before the lse write of column group 0
  __syncwarp(__activemask());
  reinterpret_cast<float4 *>(out)[i] = z;
  if (dq == 0) lse[r] = L > 0.0f ? M + logf(L) : -INFINITY;
}

}  // namespace
}  // namespace bsi

extern "C" bs_status bs_cpu_sparse_attn(const bs_dims *dims, const void *q, const bs_host_kv *kv,
                                        const bs_host_tables *tables, const int32_t *sel_idx, const int32_t *sel_cnt,
                                        float *out, float *lse, int n_threads) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!q || !kv || !kv->k_pool || !kv->v_pool || !tables || !tables->page_table || !tables->seq_lens ||
      !tables->block_tokens || !sel_idx || !sel_cnt || !out || !lse || kv->n_pages < 1 ||
      (tables->evict_bias != nullptr && tables->max_blocks_per_unit < 1))
    return BS_ERR_INVALID_ARG;
  const int units = dims->batch * dims->n_kv_heads;
  const int nt = std::max(1, std::min(n_threads, units));
  std::atomic<int> next(0);
  std::atomic<int> bad(0);
  auto work = [&]() {
    for (int u = next.fetch_add(1); u < units; u = next.fetch_add(1)) {
      const int cnt = sel_cnt[u];
      const int g = tables->block_tokens[u];
      if (cnt < 0 || cnt > dims->max_sel_per_unit || g <= 0) {
        bad.store(1);
        continue;
      }
      if (!cpu_unit(*dims, q, *tables, kv->k_pool, kv->v_pool, kv->n_pages,
                    sel_idx + static_cast<size_t>(u) * dims->max_sel_per_unit, cnt, u, out, lse))
        bad.store(1);
    }
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(work);
  work();
  for (auto &th : pool) th.join();
  return bad.load() ? BS_ERR_DEVICE_BOUNDS : BS_OK;
}

extern "C" bs_status bs_lse_merge(const bs_dims *dims, const float *out_a, const float *lse_a, const float *out_b,
                                  const float *lse_b, float *out, float *lse, bs_stream_t stream) {
  using namespace bsi;
  bs_status s = check_dims(dims);
  if (s != BS_OK) return s;
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return BS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out_a) | reinterpret_cast<uintptr_t>(out_b) | reinterpret_cast<uintptr_t>(out)) &
      15u)
    return BS_ERR_ALIGN;
  const int rows = dims->batch * dims->n_q_heads;
  const int n = rows * (dims->head_dim / 4);
  lse_merge_kernel<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      rows, dims->head_dim, out_a, lse_a, out_b, lse_b, out, lse);
  return launch_status();
}
