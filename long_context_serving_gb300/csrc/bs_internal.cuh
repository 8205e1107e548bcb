// Internal helpers shared by the kernels of libbsattn (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsattn.h"

namespace bsi {

constexpr int kPage = 16;           // tokens per physical KV page
constexpr int kMaxG = 8;            // largest GQA group handled
constexpr int kMaxBlocks = 16384;   // largest blocks-per-unit row (selection in shared memory)
constexpr int kMaxSubPerBlock = 64; // largest g/s

// ---------------------------------------------------------------------------
// Device status word: the first error code wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t *st, int code) { atomicCAS(st, 0, code); }

// ---------------------------------------------------------------------------
// Geometry of one unit at one step (forced blocks and the candidate range).
// Sink blocks [0, n_sink); local blocks [local_lo, n_blk); candidates [c_lo, c_hi).
// With local_tokens >= 1 the block holding T-1 is local, so every block below
// local_lo is complete and the candidates form one contiguous range.
// ---------------------------------------------------------------------------
struct Geom {
  int T, g, s, n_blk, n_sink, local_lo, c_lo, c_hi;
};

__host__ __device__ __forceinline__ Geom unit_geom(int T, int g, int s, int sink, int local) {
  Geom r;
  r.T = T;
  r.g = g;
  r.s = s;
  r.n_blk = (T + g - 1) / g;
  int ns = (sink + g - 1) / g;
  r.n_sink = ns < r.n_blk ? ns : r.n_blk;
  int rem = T - local;
  r.local_lo = (rem > 0 ? rem : 0) / g;
  r.c_lo = r.n_sink;
  r.c_hi = r.local_lo > r.c_lo ? r.local_lo : r.c_lo;
  return r;
}

__host__ __device__ __forceinline__ bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Rules on one unit's head configuration (documented with bs_head_cfg).
__host__ __device__ __forceinline__ bool unit_cfg_ok(int cls, int g, int s, int k, int k_e, int sink,
                                                     int local) {
  if (cls < BS_STREAMING || cls > BS_DUAL) return false;
  if (g <= 0 || g % kPage != 0 || s <= 0 || g % s != 0) return false;
  if (!is_pow2(g / s) || g / s > kMaxSubPerBlock) return false;
  if (sink < 0 || local < 1 || k < 0) return false;
  if (cls == BS_DUAL && (k_e < 0 || k_e > k)) return false;
  return true;
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk (1-D TMA) copies.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned char *align_smem_1024(unsigned char *p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation and prior generic-proxy shared accesses visible to
// the async proxy (bulk copies) before the next copy is issued.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default limit of every device-side wait (bs_set_wait_limit_ns changes it).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // one second

// Wait for a barrier phase with a wall-clock limit of limit_ns (the timer is read every
// 64 tries only). Returns false and records BS_ERR_TIMEOUT if the phase never completes.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int32_t *st,
                                                  uint64_t limit_ns = kDefaultWaitNs) {
  uint32_t n = 0;
  uint64_t t0 = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0) {
      const uint64_t t = global_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > limit_ns) {
        report(st, BS_ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Plain arrival on a barrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Barrier among `count` threads (a multiple of 32) on hardware barrier `id` (1..15;
// 0 is the one __syncthreads uses).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Global -> shared bulk copy that signals `bar` with its byte count.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// Numbers.
// ---------------------------------------------------------------------------
// bf16 pair packed in a 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float load_scalar(const void *p, size_t i, int dtype) {
  if (dtype == BS_BF16) {
    const uint16_t v = static_cast<const uint16_t *>(p)[i];
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  return static_cast<const float *>(p)[i];
}

// Order-preserving map of a float to uint32 (larger float -> larger key); -0 maps
// like +0 so that equal values tie.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of order_key.
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// ---------------------------------------------------------------------------
// Host helpers.
// ---------------------------------------------------------------------------
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every call. Returns BS_OK or the first problem.
bs_status check_dims(const bs_dims *d);

// The current limit of device-side waits in nanoseconds (bs_set_wait_limit_ns).
uint64_t wait_limit_ns();

// Tiled tensor maps over the bf16 K and V pools viewed as [n_pages * 16][head_dim]:
// boxes of 16 rows x 64 columns (128 bytes) with 128-byte swizzle.
bs_status make_kv_tensor_maps(const bs_dims &d, const bs_kv &kv, CUtensorMap *tk, CUtensorMap *tv);

// Dynamic shared memory is re-based to a 1024-byte boundary (the 128-byte swizzle
// atom of TMA copies); kernels that need it allocate this much more.
constexpr int kSmemAlignSlack = 1024;

inline bs_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}

}  // namespace bsi
