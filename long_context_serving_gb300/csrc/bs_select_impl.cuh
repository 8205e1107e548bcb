// Device code of the per-unit block selection (a3) and set-difference (a5), shared by
// the stand-alone kernels and the fused decode step.
//
// Selection: "Technische Samenvatting: Fluxion", Kerninzichten item 2 (streaming vs
// retrieval heads); "Technisches Resümee: NOSA", Methodik / 1. Algorithmus: NOSA,
// "Dual-Selection-Mechanismus" and "ED-DMA". Set-difference: NOSA, "2. System: NOSI".
//
// Keys are float32 values mapped to order-preserving uint32; ties go to the lowest
// block index and every selection is written in ascending order, so nothing is sorted.
// Two implementations of the same selection:
//   * select_unit_regs (units with at most 32 candidates per thread, every workload
//     here): candidates in registers, striped over the threads; top-k by refining a
//     2048-bucket histogram level by level; output order by ballot-ranked compaction;
//   * select_unit_flags + compact_selection (larger units): keys and flags in shared
//     memory; top-k by one min/max pass, a 2048-bucket histogram and an exact ranking of
//     the boundary bucket (topk_mark), with a four-pass 8-bit radix select for heavy
//     ties (topk_mark_radix); compaction over block indices.
// select_unit picks one. Set-difference after a selection: setdiff_sorted.
#pragma once

#include "bs_internal.cuh"

namespace bsi {

// flag bits per block
constexpr uint8_t kSel = 1;     // in the final selection
constexpr uint8_t kAlive = 2;   // eligible for Gamma_e (dual)
constexpr uint8_t kEvict = 4;   // chosen by Gamma_e
constexpr uint8_t kElig = 8;    // eligible in the current top-k pass

constexpr uint8_t kBnd = 16;    // in the boundary bucket of the fast top-k
constexpr int kBuckets = 2048;  // histogram buckets of the fast top-k
constexpr int kBndDirect = 256; // boundary buckets up to this size are ranked directly

template <int NT>
struct __align__(16) SelShared {  // hist is cleared with 16-byte stores
  static constexpr int kWarps = NT / 32;
  uint32_t hist[kBuckets];      // the radix passes use the first 256
  int warp_tot[kWarps];
  int wt[2][kWarps];            // warp totals of the one-barrier scan, two buffers
  int wt2[2][kWarps];           // their inclusive prefix (CTAs of more than 8 warps)
  uint32_t warp_min[kWarps], warp_max[kWarps];
  int warp_cnt[kWarps];
  uint32_t mm[4];               // CTA-wide min, max, count (CTAs of more than 8 warps)
  int bcast[4];
  int bnd_n;
  int bnd_idx[kBndDirect];
  int ord[NT];                  // per (round, warp) counts of the ordered ranking
  int ord2[NT];                 // their exclusive prefix
};

__device__ __forceinline__ bool sorted_contains(const int32_t *v, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo < n && v[lo] == x;
}

static_assert(alignof(SelShared<256>) >= 16 && alignof(SelShared<512>) >= 16, "16-byte stores into hist");

// Exclusive prefix sum of one int per thread over the CTA; *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, SelShared<NT> &sh, int *total) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < W ? sh.warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < W) sh.warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = (warp > 0 ? sh.warp_tot[warp - 1] : 0) + x - v;
  *total = sh.warp_tot[W - 1];
  __syncthreads();
  return before;
}

// Marks with `mark` the k blocks of [lo, hi) carrying `elig` with the largest keys
// (keys[c - lo]), lower index first among equal keys. Four-pass 8-bit radix select.
template <int NT>
__device__ __noinline__ void topk_mark_radix(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k,
                                             uint8_t mark, SelShared<NT> &sh, uint8_t elig = kElig) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  // Contiguous per-thread ranges keep the index order for the tie pass.
  const int per = (n + NT - 1) / NT;
  const int a = lo + tid * per, e = min(hi, a + per);
  int my = 0;
  for (int c = a; c < e; ++c) my += (flags[c] & elig) ? 1 : 0;
  int n_elig;
  block_excl_scan<NT>(my, sh, &n_elig);
  if (k >= n_elig) {
    for (int c = a; c < e; ++c)
      if (flags[c] & elig) flags[c] |= mark;
    __syncthreads();
    return;
  }
  uint32_t prefix = 0, pmask = 0;
  int rem = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) sh.hist[i] = 0;
    __syncthreads();
    for (int base = lo; base < hi; base += NT) {
      const int c = base + tid;
      bool valid = false;
      uint32_t digit = 256;
      if (c < hi && (flags[c] & elig)) {
        const uint32_t key = keys[c - lo];
        if ((key & pmask) == prefix) {
          valid = true;
          digit = (key >> shift) & 255u;
        }
      }
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (valid && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins [255-8l-7, 255-8l], scanned from the top.
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) cnt += static_cast<int>(sh.hist[255 - 8 * lane - i]);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int before = incl - cnt;
      if (before < rem && rem <= incl) {
        int run = before;
        for (int i = 0; i < 8; ++i) {
          const int bin = 255 - 8 * lane - i;
          const int h = static_cast<int>(sh.hist[bin]);
          if (run + h >= rem) {
            sh.bcast[0] = bin;
            sh.bcast[1] = rem - run;
            break;
          }
          run += h;
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sh.bcast[0]) << shift;
    pmask |= 255u << shift;
    rem = sh.bcast[1];
    __syncthreads();
  }
  // prefix is the k-th largest key; `rem` of the keys equal to it are taken.
  int eq = 0;
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & elig)) continue;
    const uint32_t key = keys[c - lo];
    if (key > prefix) flags[c] |= mark;
    else if (key == prefix) ++eq;
  }
  int tot;
  int rank = block_excl_scan<NT>(eq, sh, &tot);
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & elig) || keys[c - lo] != prefix) continue;
    if (rank < rem) flags[c] |= mark;
    ++rank;
  }
  __syncthreads();
}

// Marks with `mark` the k blocks of [lo, hi) carrying kElig with the largest keys
// (keys[c - lo]), lower index first among equal keys; the same result as
// topk_mark_radix with fewer CTA barriers:
//   1. min, max and count of the eligible keys (one barrier);
//   2. a histogram over 2048 buckets of the float value placed linearly between the
//      minimum and the maximum, (x - min) * (2048 / (max - min)) in fp32 with round to
//      nearest: subtraction, multiplication by a positive constant and truncation are
//      each monotone, so every key in a bucket above the boundary bucket B is taken
//      and every key below is not;
//   3. a suffix count over the buckets finds B and how many of its keys are taken;
//   4. keys in B are ranked exactly by (key desc, index asc): directly when B holds
//      at most 256 keys, otherwise by the radix select restricted to B.
template <int NT>
__device__ __noinline__ void topk_mark(const uint32_t *keys, uint8_t *flags, int lo, int hi, int k, uint8_t mark,
                                       SelShared<NT> &sh) {
  constexpr int W = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = hi - lo;
  if (k <= 0 || n <= 0) return;
  const int per = (n + NT - 1) / NT;
  const int a = lo + tid * per, e = min(hi, a + per);
  // 1. min / max / count
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  int cnt = 0;
  for (int c = a; c < e; ++c)
    if (flags[c] & kElig) {
      const uint32_t key = keys[c - lo];
      kmin = min(kmin, key);
      kmax = max(kmax, key);
      ++cnt;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if (lane == 0) {
    sh.warp_min[warp] = kmin;
    sh.warp_max[warp] = kmax;
    sh.warp_cnt[warp] = cnt;
  }
  for (int i = tid; i < kBuckets; i += NT) sh.hist[i] = 0;
  if (tid == 0) sh.bnd_n = 0;
  __syncthreads();
  kmin = 0xffffffffu;
  kmax = 0u;
  int n_elig = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    kmin = min(kmin, sh.warp_min[w]);
    kmax = max(kmax, sh.warp_max[w]);
    n_elig += sh.warp_cnt[w];
  }
  if (k >= n_elig || kmin == kmax) {
    // Everything is taken, or every key ties: the radix select settles it cheaply.
    topk_mark_radix<NT>(keys, flags, lo, hi, k, mark, sh);
    return;
  }
  // 2. histogram of the monotone bucket map
  // A zero, infinite or NaN range (equal keys, infinities) puts every key in bucket 0,
  // which the exact rank below still orders correctly.
  const float xmin = key_value(kmin);
  const float range = key_value(kmax) - xmin;
  float bscale = (range > 0.0f && range <= 3.0e38f) ? static_cast<float>(kBuckets) / range : 0.0f;
  if (!(bscale <= 3.0e38f)) bscale = 0.0f;  // a subnormal range
  auto bucket = [&](uint32_t key) -> uint32_t {
    if (bscale == 0.0f) return 0u;
    const float f = (key_value(key) - xmin) * bscale;  // in [0, 2048 (1 + eps)]
    return f >= static_cast<float>(kBuckets - 1) ? static_cast<uint32_t>(kBuckets - 1) : static_cast<uint32_t>(f);
  };
  for (int c = a; c < e; ++c)
    if (flags[c] & kElig) atomicAdd(&sh.hist[bucket(keys[c - lo])], 1u);
  __syncthreads();
  // 3. thread t owns buckets [kBuckets - bpt (t + 1), kBuckets - bpt t): suffix counts
  constexpr int bpt = kBuckets / NT;
  const int top = kBuckets - bpt * tid - 1;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < bpt; ++i) mine += static_cast<int>(sh.hist[top - i]);
  int total;
  const int above = block_excl_scan<NT>(mine, sh, &total);
  if (above < k && k <= above + mine) {
    int run = above;
    for (int i = 0; i < bpt; ++i) {
      const int hcount = static_cast<int>(sh.hist[top - i]);
      if (run + hcount >= k) {
        sh.bcast[0] = top - i;    // boundary bucket B
        sh.bcast[1] = k - run;    // keys of B to take
        sh.bcast[2] = hcount;     // keys in B
        break;
      }
      run += hcount;
    }
  }
  __syncthreads();
  const uint32_t B = static_cast<uint32_t>(sh.bcast[0]);
  const int rem = sh.bcast[1], in_b = sh.bcast[2];
  // 4. take the buckets above B; collect B
  for (int c = a; c < e; ++c) {
    if (!(flags[c] & kElig)) continue;
    const uint32_t bk = bucket(keys[c - lo]);
    if (bk > B) flags[c] |= mark;
    else if (bk == B) {
      if (in_b <= kBndDirect) sh.bnd_idx[atomicAdd(&sh.bnd_n, 1)] = c;
      else flags[c] |= kBnd;
    }
  }
  __syncthreads();
  if (in_b <= kBndDirect) {
    for (int i = tid; i < in_b; i += NT) {
      const int c = sh.bnd_idx[i];
      const uint32_t key = keys[c - lo];
      int rank = 0;
      for (int j = 0; j < in_b; ++j) {
        const int c2 = sh.bnd_idx[j];
        const uint32_t k2 = keys[c2 - lo];
        rank += (k2 > key || (k2 == key && c2 < c)) ? 1 : 0;
      }
      if (rank < rem) flags[c] |= mark;
    }
    __syncthreads();
  } else {
    topk_mark_radix<NT>(keys, flags, lo, hi, rem, mark, sh, kBnd);
    for (int c = a; c < e; ++c) flags[c] &= static_cast<uint8_t>(~kBnd);
    __syncthreads();
  }
}

// Per-unit inputs of the selection.
struct SelUnit {
  int cls, k, k_e;
  Geom ge;
  const float *scores;   // row of unit u (candidates [c_lo, c_hi) are read)
  const float *evict;    // row of unit u, dual only
  uint8_t *alive;        // row of unit u, dual only
};

// Selects the blocks of one unit into `flags[0, n_blk)` (bit kSel). Uses keys[n_blk]
// and flags[n_blk] in shared memory. Reads scores with L2-only loads so that values
// written by other CTAs of the same grid are seen. All NT threads must call it.
template <int NT>
__device__ __noinline__ void select_unit_flags(const SelUnit &su, uint32_t *keys, uint8_t *flags, SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const Geom &ge = su.ge;
  const int lo = ge.c_lo, hi = ge.c_hi;
  for (int c = tid; c < ge.n_blk; c += NT) {
    const bool forced = c < ge.n_sink || c >= ge.local_lo;
    uint8_t f = forced ? kSel : 0;
    if (su.cls == BS_DUAL && c >= lo && c < hi && su.alive[c]) f |= kAlive;
    flags[c] = f;
  }
  __syncthreads();
  if (su.cls == BS_RETRIEVAL) {
    for (int c = lo + tid; c < hi; c += NT) {
      keys[c - lo] = order_key(__ldcg(su.scores + c));
      flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k, kSel, sh);
  } else if (su.cls == BS_DUAL) {
    // Gamma_e: the k_e largest eviction logits among alive candidates.
    for (int c = lo + tid; c < hi; c += NT) {
      keys[c - lo] = order_key(su.evict[c]);
      if (flags[c] & kAlive) flags[c] |= kElig;
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k_e, kEvict, sh);
    // Strict eviction: candidates outside Gamma_e are dead from now on. Gamma_q: the
    // k - k_e largest scores among the candidates outside Gamma_e.
    for (int c = lo + tid; c < hi; c += NT) {
      const uint8_t f = flags[c];
      su.alive[c] = (f & kEvict) ? 1 : 0;
      keys[c - lo] = order_key(__ldcg(su.scores + c));
      flags[c] = static_cast<uint8_t>(((f & kEvict) ? kSel : kElig) | (f & kEvict));
    }
    __syncthreads();
    topk_mark<NT>(keys, flags, lo, hi, su.k - su.k_e, kSel, sh);
  }
}

// Ascending compaction of the flagged blocks into out[0, cap) (-1 padded) and, if
// given, into the shared list `copy`. Returns the count, or -1 when it exceeds cap
// (then the row is all -1).
template <int NT>
__device__ __noinline__ int compact_selection(const uint8_t *flags, int n_blk, int32_t *out, int cap, int32_t *copy,
                                 SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const int per = (n_blk + NT - 1) / NT;
  const int a = tid * per, e = min(n_blk, a + per);
  int mine = 0;
  for (int c = a; c < e; ++c) mine += (flags[c] & kSel) ? 1 : 0;
  int total;
  int pos = block_excl_scan<NT>(mine, sh, &total);
  if (total > cap) {
    for (int i = tid; i < cap; i += NT) out[i] = -1;
    return -1;
  }
  for (int c = a; c < e; ++c)
    if (flags[c] & kSel) {
      out[pos] = c;
      if (copy) copy[pos] = c;
      ++pos;
    }
  for (int i = total + tid; i < cap; i += NT) out[i] = -1;
  return total;
}

// ---------------------------------------------------------------------------
// Register-resident selection (units with at most NT * R candidates).
//
// Candidate c = c_lo + i * NT + t is element i of thread t: the loads of scores and
// logits are coalesced, every per-candidate decision is a bit of a per-thread mask,
// and shared memory holds only a histogram and a few reduction slots. The top-k refines
// a 2048-bucket histogram level by level (linear float buckets first, then integer
// buckets on the order keys, each level shrinking the key range of the boundary bucket
// by 2^11) until the boundary bucket is taken whole or all its keys are equal; equal
// keys go to the lowest block index. The output order is ascending block index: a
// ranking of the taken candidates by ballots per (round, warp) and one prefix scan.
// ---------------------------------------------------------------------------

// Exclusive prefix sum over the CTA. Up to 8 warps: one barrier, after which every
// thread adds the warp totals itself; two consecutive calls with the same `buf` need a
// barrier between them. More warps: warp 0 scans the warp totals between two barriers
// (every thread then reads two values instead of one per warp). *total gets the sum.
template <int NT>
__device__ __forceinline__ int block_scan1(int v, SelShared<NT> &sh, int buf, int *total) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.wt[buf][warp] = x;
  __syncthreads();
  int off = 0, tot = 0;
  if constexpr (W <= 8) {
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const int t = sh.wt[buf][w];
      off += w < warp ? t : 0;
      tot += t;
    }
  } else {
    if (warp == 0) {
      int w = lane < W ? sh.wt[buf][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < W) sh.wt2[buf][lane] = w;   // inclusive
    }
    __syncthreads();
    off = warp > 0 ? sh.wt2[buf][warp - 1] : 0;
    tot = sh.wt2[buf][W - 1];
  }
  *total = tot;
  return off + x - v;
}

// CTA-wide min, max and sum (results in every thread): one barrier up to 8 warps, two
// beyond (warp 0 reduces the warp values).
template <int NT>
__device__ __forceinline__ void block_min_max_count(uint32_t &kmin, uint32_t &kmax, int &cnt, SelShared<NT> &sh) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  cnt = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<uint32_t>(cnt)));
  if (lane == 0) {
    sh.warp_min[warp] = kmin;
    sh.warp_max[warp] = kmax;
    sh.warp_cnt[warp] = cnt;
  }
  __syncthreads();
  if constexpr (W <= 8) {
    kmin = 0xffffffffu;
    kmax = 0u;
    cnt = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      kmin = min(kmin, sh.warp_min[w]);
      kmax = max(kmax, sh.warp_max[w]);
      cnt += sh.warp_cnt[w];
    }
  } else {
    if (warp == 0) {
      const uint32_t a = __reduce_min_sync(0xffffffffu, lane < W ? sh.warp_min[lane] : 0xffffffffu);
      const uint32_t b = __reduce_max_sync(0xffffffffu, lane < W ? sh.warp_max[lane] : 0u);
      const uint32_t n = __reduce_add_sync(0xffffffffu, lane < W ? static_cast<uint32_t>(sh.warp_cnt[lane]) : 0u);
      if (lane == 0) {
        sh.mm[0] = a;
        sh.mm[1] = b;
        sh.mm[2] = n;
      }
    }
    __syncthreads();
    kmin = sh.mm[0];
    kmax = sh.mm[1];
    cnt = static_cast<int>(sh.mm[2]);
  }
}

// Rank of each set bit of `bits` among the set bits of the whole CTA in ascending
// candidate order (rank[i] is valid where bit i is set). Returns the number of set bits.
template <int NT, int R>
__device__ __forceinline__ int ordered_ranks(uint32_t bits, int nr, int (&rank)[R], SelShared<NT> &sh) {
  constexpr int W = NT / 32;
  static_assert(R * W <= NT, "one scan slot per (round, warp)");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    rank[i] = 0;
    if (i < nr) {
      const uint32_t m = __ballot_sync(0xffffffffu, (bits >> i) & 1u);
      rank[i] = __popc(m & lt);
      if (lane == 0) sh.ord[i * W + warp] = __popc(m);
    }
  }
  __syncthreads();
  int total;
  const int ex = block_scan1<NT>(threadIdx.x < nr * W ? sh.ord[threadIdx.x] : 0, sh, 0, &total);
  sh.ord2[threadIdx.x] = ex;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < R; ++i)
    if (i < nr) rank[i] += sh.ord2[i * W + warp];
  return total;
}

// The k largest keys among the elements flagged in `elig` (lowest candidate index
// first among equal keys); returns them as a mask. All threads call it with the same
// nr and k.
template <int NT, int R>
__device__ __forceinline__ uint32_t topk_regs(const uint32_t (&key)[R], uint32_t elig, int nr, int k,
                                              SelShared<NT> &sh) {
  constexpr int bpt = kBuckets / NT;  // buckets per thread in the boundary search
  const int tid = threadIdx.x;
  uint32_t take = 0u, E = elig;
  int need = k;
  bool done = need <= 0;
  __syncthreads();  // earlier readers of the reduction slots and the histogram are done
  for (int level = 0; level < 6 && !done; ++level) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (i < nr && ((E >> i) & 1u)) {
        kmin = min(kmin, key[i]);
        kmax = max(kmax, key[i]);
        ++cnt;
      }
    for (int j = tid; j < kBuckets / 4; j += NT) reinterpret_cast<uint4 *>(sh.hist)[j] = make_uint4(0u, 0u, 0u, 0u);
    block_min_max_count<NT>(kmin, kmax, cnt, sh);
    if (need >= cnt) {
      take |= E;
      done = true;
      break;
    }
    if (kmin == kmax) break;  // all equal: lowest indices, below
    // Monotone bucket map: linear in the float value on the first level when the
    // range is finite and normal, otherwise (key - kmin) >> shift.
    const float xmin = key_value(kmin);
    const float range = key_value(kmax) - xmin;
    float bscale = (level == 0 && range > 0.0f && range <= 3.0e38f) ? static_cast<float>(kBuckets) / range : 0.0f;
    if (!(bscale <= 3.0e38f)) bscale = 0.0f;
    const uint32_t span = kmax - kmin;
    const int bits = 32 - __clz(span);
    const int shift = bits > 11 ? bits - 11 : 0;
    auto bucket = [&](uint32_t kk) -> uint32_t {
      if (bscale > 0.0f) {
        // f in [0, 2048 (1 + eps)]; adding 2^23 rounds it to an integer in the low
        // mantissa bits (monotone, like every step here).
        const float f = (key_value(kk) - xmin) * bscale;
        const uint32_t rb = __float_as_uint(f + 8388608.0f) - 0x4B000000u;
        return min(rb, static_cast<uint32_t>(kBuckets - 1));
      }
      return (kk - kmin) >> shift;
    };
    constexpr bool kCache = R <= 8;  // bucket of each element kept in registers
    uint32_t bkc[kCache ? R : 1];
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (i < nr && ((E >> i) & 1u)) {
        const uint32_t bk = bucket(key[i]);
        if (kCache) bkc[kCache ? i : 0] = bk;
        atomicAdd(&sh.hist[bk], 1u);
      }
    __syncthreads();
    // Thread t owns buckets [kBuckets - bpt (t + 1), kBuckets - bpt t), highest first.
    const int top = kBuckets - bpt * tid - 1;
    int hc[bpt];
    int mine = 0;
#pragma unroll
    for (int j = 0; j < bpt; ++j) {
      hc[j] = static_cast<int>(sh.hist[top - j]);
      mine += hc[j];
    }
    int tot;
    const int above = block_scan1<NT>(mine, sh, level & 1, &tot);
    if (above < need && need <= above + mine) {
      int run = above;
#pragma unroll
      for (int j = 0; j < bpt; ++j) {
        if (run + hc[j] >= need) {
          sh.bcast[0] = top - j;    // boundary bucket
          sh.bcast[1] = need - run; // keys of it to take
          sh.bcast[2] = hc[j];      // keys in it
          break;
        }
        run += hc[j];
      }
    }
    __syncthreads();
    const uint32_t B = static_cast<uint32_t>(sh.bcast[0]);
    const int rem = sh.bcast[1], in_b = sh.bcast[2];
    uint32_t nextE = 0u;
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (i < nr && ((E >> i) & 1u)) {
        const uint32_t bk = kCache ? bkc[kCache ? i : 0] : bucket(key[i]);
        if (bk > B) take |= 1u << i;
        else if (bk == B) nextE |= 1u << i;
      }
    E = nextE;
    need = rem;
    if (rem == in_b) {
      take |= E;
      done = true;
    }
  }
  if (!done) {
    // Every remaining key is equal (or the level bound was reached): take the `need`
    // lowest candidate indices of E.
    int rank[R];
    ordered_ranks<NT, R>(E, nr, rank, sh);
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (i < nr && ((E >> i) & 1u) && rank[i] < need) take |= 1u << i;
  }
  return take;
}

// Selects the blocks of one unit (at most NT * R candidates) and writes them ascending
// to out[0, cap) (-1 padded) and, if given, to `copy`. Dual units also update their
// alive row. Returns the count, or -1 when it exceeds cap (the row is then all -1).
// Reads scores with L2-only loads so that values written by other CTAs of the same grid
// are seen. All NT threads call it.
template <int NT, int R>
__device__ __forceinline__ int select_unit_regs(const SelUnit &su, int32_t *out, int cap, int32_t *copy,
                                                SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const Geom ge = su.ge;
  const int lo = ge.c_lo, hi = ge.c_hi;
  const int nr = (hi - lo + NT - 1) / NT;
  uint32_t valid = 0u;
#pragma unroll
  for (int i = 0; i < R; ++i)
    if (i < nr && lo + i * NT + tid < hi) valid |= 1u << i;
  uint32_t take = 0u;
  const int passes = su.cls == BS_DUAL ? 2 : (su.cls == BS_RETRIEVAL ? 1 : 0);
  for (int p = 0; p < passes; ++p) {
    // Dual: pass 0 is Gamma_e on the eviction logits among alive candidates; pass 1 is
    // Gamma_q on the scores among the candidates outside Gamma_e. Retrieval: scores.
    const bool gamma_e = su.cls == BS_DUAL && p == 0;
    uint32_t key[R];
    uint32_t elig = 0u;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      key[i] = 0u;
      if ((valid >> i) & 1u) {
        const int c = lo + i * NT + tid;
        if (gamma_e) {
          key[i] = order_key(su.evict[c]);
          if (su.alive[c]) elig |= 1u << i;
        } else {
          key[i] = order_key(__ldcg(su.scores + c));
          if (!((take >> i) & 1u)) elig |= 1u << i;
        }
      }
    }
    const int kk = gamma_e ? su.k_e : (su.cls == BS_DUAL ? su.k - su.k_e : su.k);
    const uint32_t t = topk_regs<NT, R>(key, elig, nr, kk, sh);
    if (gamma_e) {
      // Strict eviction: candidates outside Gamma_e are dead from now on.
#pragma unroll
      for (int i = 0; i < R; ++i)
        if ((valid >> i) & 1u) su.alive[lo + i * NT + tid] = static_cast<uint8_t>((t >> i) & 1u);
    }
    take |= t;
  }
  // Ascending output: sink blocks [0, c_lo), the taken candidates, local blocks [c_hi, n_blk).
  int rank[R];
  const int n_take = passes > 0 ? ordered_ranks<NT, R>(take, nr, rank, sh) : 0;
  const int n_local = ge.n_blk - hi;
  const int total = lo + n_take + n_local;
  if (total > cap) {
    for (int i = tid; i < cap; i += NT) out[i] = -1;
    return -1;
  }
  for (int c = tid; c < lo; c += NT) {
    out[c] = c;
    if (copy) copy[c] = c;
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
    if ((take >> i) & 1u) {
      const int pos = lo + rank[i], c = lo + i * NT + tid;
      out[pos] = c;
      if (copy) copy[pos] = c;
    }
  for (int j = tid; j < n_local; j += NT) {
    const int pos = lo + n_take + j;
    out[pos] = hi + j;
    if (copy) copy[pos] = hi + j;
  }
  for (int i = total + tid; i < cap; i += NT) out[i] = -1;
  return total;
}

// Selection of one unit into out[0, cap) (and `copy`): the register-resident path up
// to NT * 32 candidates (NT * 8 for CTAs of 1024 threads), otherwise flags and keys in
// shared memory (keys[n_blk], flags[n_blk]). Returns the count, or -1 when it exceeds
// cap.
template <int NT>
__device__ __forceinline__ int select_unit(const SelUnit &su, uint32_t *keys, uint8_t *flags, int32_t *out, int cap,
                                           int32_t *copy, SelShared<NT> &sh) {
  const int nr = (su.ge.c_hi - su.ge.c_lo + NT - 1) / NT;
  if (nr <= 4) return select_unit_regs<NT, 4>(su, out, cap, copy, sh);
  if (NT >= 1024) {
    // (1024 threads: registers for up to 8 candidates a thread, the shared-memory path
    // beyond)
    if (nr <= 8) return select_unit_regs<NT, (NT >= 1024 ? 8 : 32)>(su, out, cap, copy, sh);
  } else if (nr <= 32) {
    return select_unit_regs<NT, (NT >= 1024 ? 8 : 32)>(su, out, cap, copy, sh);
  }
  select_unit_flags<NT>(su, keys, flags, sh);
  return compact_selection<NT>(flags, su.ge.n_blk, out, cap, copy, sh);
}

// Set-difference of two ascending lists in shared memory (cur[0, nc), prev[0, np)):
// added = cur \ prev and removed = prev \ cur, ascending, -1 padded to cap. Membership by
// binary search; one packed scan orders both outputs. All NT threads call it.
template <int NT>
__device__ __forceinline__ int2 setdiff_sorted(const int32_t *cur, int nc, const int32_t *prev, int np,
                                               int32_t *added, int32_t *removed, int cap, SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const int pc = (nc + NT - 1) / NT, pp = (np + NT - 1) / NT;
  const int ca = tid * pc, ce = min(nc, ca + pc);
  const int pa = tid * pp, pe = min(np, pa + pp);
  int na = 0, nr = 0;
  for (int i = ca; i < ce; ++i) na += sorted_contains(prev, np, cur[i]) ? 0 : 1;
  for (int i = pa; i < pe; ++i) nr += sorted_contains(cur, nc, prev[i]) ? 0 : 1;
  int total;
  const int packed = block_scan1<NT>((na << 16) | nr, sh, 1, &total);
  int wa = packed >> 16, wr = packed & 0xffff;
  for (int i = ca; i < ce; ++i)
    if (!sorted_contains(prev, np, cur[i])) added[wa++] = cur[i];
  for (int i = pa; i < pe; ++i)
    if (!sorted_contains(cur, nc, prev[i])) removed[wr++] = prev[i];
  const int ta = total >> 16, tr = total & 0xffff;
  for (int i = ta + tid; i < cap; i += NT) added[i] = -1;
  for (int i = tr + tid; i < cap; i += NT) removed[i] = -1;
  return make_int2(ta, tr);
}

// ---------------------------------------------------------------------------
// Set-difference of two ascending lists held in shared memory.
// ---------------------------------------------------------------------------

// Writes the elements of a[0..na) missing from b[0..nb) to dst (ascending), pads
// with -1 up to cap and returns the count. All NT threads must call it.
template <int NT>
__device__ int sorted_diff_into(const int32_t *a, int na, const int32_t *b, int nb, int32_t *dst, int cap,
                                SelShared<NT> &sh) {
  const int tid = threadIdx.x;
  const int per = (na + NT - 1) / NT;
  const int s = tid * per, e = min(na, s + per);
  int mine = 0;
  for (int i = s; i < e; ++i) mine += sorted_contains(b, nb, a[i]) ? 0 : 1;
  int total;
  int before = block_excl_scan<NT>(mine, sh, &total);
  for (int i = s; i < e; ++i)
    if (!sorted_contains(b, nb, a[i])) dst[before++] = a[i];
  for (int i = total + tid; i < cap; i += NT) dst[i] = -1;
  return total;
}

}  // namespace bsi
