// Device building blocks for the selector: mbarriers, bulk copies, named
// barriers, Philox4x32-10, the float order key and bitonic networks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace topk {

// ---------------------------------------------------------------------------
// Shared-memory mbarriers and bulk copies (inline PTX, sm_90+ forms).

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the phase did not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bounded wait that sleeps `ns` nanoseconds between polls, so that a warp
// waiting for a long time leaves the issue slots of its SM sub-partition to
// the warps that have work.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t limit,
                                                unsigned ns) {
  for (uint32_t it = 0; it < limit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(ns);
  }
  return false;
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`.  Both
// addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// An L2 policy that evicts first: for data read once (a stream must not push
// the kernel's code and small shared words out of L2).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_load with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (sm_90+).  A grid launched with programmatic
// stream serialization may start while the grid before it in the stream is
// still running; grid_dep_wait() blocks the calling thread until that grid has
// completed and its memory is visible, so every thread calls it before it
// touches global memory another grid may write.  grid_dep_launch() lets the
// next such grid be scheduled on SMs this one leaves free.

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// A team of NT threads that synchronises on named barrier BAR.

template <int NT, int BAR>
struct Team {
  static constexpr int size = NT;
  static __device__ __forceinline__ void sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
  }
  // Barrier that also returns whether any thread passed `v` true.
  static __device__ __forceinline__ bool sync_or(bool v) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(out)
        : "r"(uint32_t(v)), "n"(BAR), "n"(NT)
        : "memory");
    return out != 0;
  }
};

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32
// multiplies with the high halves xor-ed into the other words and the key.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// ---------------------------------------------------------------------------
// Order key: a monotone map of float bits to uint32 (the unsigned order of the
// keys is the value order, with -0.0 below +0.0).

__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return bits ^ (uint32_t(int32_t(bits) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t key) {
  const uint32_t bits = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(bits);
}

// The smallest float whose key is >= the threshold word's key; -inf while the
// threshold is still the empty word 0.
__device__ __forceinline__ float threshold_float(uint64_t th) {
  const uint32_t hi = uint32_t(th >> 32);
  return hi < 0x007FFFFFu ? -__int_as_float(0x7F800000) : key_to_float(hi);
}

__device__ __forceinline__ int next_pow2_dev(int x) {
  return x <= 1 ? 1 : 1 << (32 - __clz(x - 1));
}

// ---------------------------------------------------------------------------
// Bitonic networks (Batcher) over shared arrays whose size is a power of two.
// `t` is the caller's index within team T.  Each ends with a team barrier.

// Sort descending.
template <class T>
__device__ void bitonic_sort_desc(uint64_t* a, int n, int t) {
  const int half = n >> 1;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int u = t; u < half; u += T::size) {
        const int i = 2 * u - (u & (stride - 1));
        const int j = i + stride;
        const uint64_t x = a[i], y = a[j];
        const bool desc = (i & size) == 0;
        if ((x < y) == desc) {
          a[i] = y;
          a[j] = x;
        }
      }
      T::sync();
    }
  }
}

// Sort descending a set of `nseq` bitonic sequences of length n, the q-th
// starting at a + q * gap.
template <class T>
__device__ void bitonic_merge_desc_multi(uint64_t* a, int n, int nseq, int gap, int t) {
  const int half = n >> 1;
  const int work = half * nseq;
  for (int stride = half; stride > 0; stride >>= 1) {
    for (int u = t; u < work; u += T::size) {
      const int q = u / half;
      const int v = u - q * half;
      uint64_t* b = a + q * gap;
      const int i = 2 * v - (v & (stride - 1));
      const int j = i + stride;
      const uint64_t x = b[i], y = b[j];
      if (x < y) {
        b[i] = y;
        b[j] = x;
      }
    }
    T::sync();
  }
}

// Sort ascending (u32 keys).
template <class T>
__device__ void bitonic_sort_asc_u32(uint32_t* a, int n, int t) {
  const int half = n >> 1;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int u = t; u < half; u += T::size) {
        const int i = 2 * u - (u & (stride - 1));
        const int j = i + stride;
        const uint32_t x = a[i], y = a[j];
        const bool asc = (i & size) == 0;
        if ((x > y) == asc) {
          a[i] = y;
          a[j] = x;
        }
      }
      T::sync();
    }
  }
}


// Register-resident bitonic sort, descending, of N = T::size * E words: team
// thread t holds words t*E .. t*E+E-1 in v[] on entry and on exit.  Strides
// below E stay in registers, strides below 32*E move between lanes with
// shuffles, and only the widest strides go through shared memory, alternating
// between buf0 and buf1 (N words each) so each such stage needs one barrier.
// The caller must make sure no thread still reads buf0/buf1 on entry.
template <int E, int STRIDE>
__device__ __forceinline__ void cas_in_regs(uint64_t (&v)[E], int base, int size) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e & STRIDE) == 0) {
      const bool desc = ((base + e) & size) == 0;
      const uint64_t a = v[e], b = v[e + STRIDE];
      const bool sw = desc ? (a < b) : (a > b);
      v[e] = sw ? b : a;
      v[e + STRIDE] = sw ? a : b;
    }
  }
}

template <class T, int E>
__device__ __forceinline__ void bitonic_sort_regs(uint64_t (&v)[E], int t, uint64_t* buf0, uint64_t* buf1) {
  constexpr int N = T::size * E;
  const int base = t * E;
  int flip = 0;
  for (int size = 2; size <= N; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < E) {
        if constexpr (E > 1) { if (stride == 1) cas_in_regs<E, 1>(v, base, size); }
        if constexpr (E > 2) { if (stride == 2) cas_in_regs<E, (E > 2 ? 2 : 1)>(v, base, size); }
        if constexpr (E > 4) { if (stride == 4) cas_in_regs<E, (E > 4 ? 4 : 1)>(v, base, size); }
        if constexpr (E > 8) { if (stride == 8) cas_in_regs<E, (E > 8 ? 8 : 1)>(v, base, size); }
      } else if (stride < 32 * E) {
        const int lm = stride / E;
        const bool lower = (base & stride) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t p = __shfl_xor_sync(0xFFFFFFFFu, v[e], lm);
          const bool desc = ((base + e) & size) == 0;
          const bool keep_max = lower == desc;
          const bool take = keep_max ? (p > v[e]) : (p < v[e]);
          v[e] = take ? p : v[e];
        }
      } else {
        uint64_t* buf = flip ? buf1 : buf0;
        flip ^= 1;
#pragma unroll
        for (int e = 0; e < E; ++e) buf[base + e] = v[e];
        T::sync();
        const bool lower = (base & stride) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t p = buf[(base + e) ^ stride];
          const bool desc = ((base + e) & size) == 0;
          const bool keep_max = lower == desc;
          const bool take = keep_max ? (p > v[e]) : (p < v[e]);
          v[e] = take ? p : v[e];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Grouped bitonic network.  Each barrier round applies up to three
// consecutive strides of one merge level: a thread loads the 2, 4 or 8
// elements that those strides connect (indices base + c * lo), runs the
// compare-exchanges in registers and stores them back.  A 512-word sort takes
// 18 barrier rounds instead of 45 single-stride stages.

template <int NS, typename K>
__device__ __forceinline__ void bitonic_group(K* a, int base, int lo, bool larger_first) {
  constexpr int G = 1 << NS;
  K v[G];
#pragma unroll
  for (int c = 0; c < G; ++c) v[c] = a[base + c * lo];
#pragma unroll
  for (int j = NS - 1; j >= 0; --j) {
#pragma unroll
    for (int c = 0; c < G; ++c) {
      if (!((c >> j) & 1)) {
        const K x = v[c], y = v[c | (1 << j)];
        const bool sw = larger_first ? (x < y) : (x > y);
        v[c] = sw ? y : x;
        v[c | (1 << j)] = sw ? x : y;
      }
    }
  }
#pragma unroll
  for (int c = 0; c < G; ++c) a[base + c * lo] = v[c];
}

// Bitonic network over `nseq` arrays of n (a power of two) elements, the q-th
// at a + q * gap, from merge level `first_size` up to n: first_size = 2 sorts,
// first_size = n sorts a bitonic input (a merge).  DESC: largest first.
// Ends with a team barrier.
template <class T, typename K, bool DESC>
__device__ void bitonic_network(K* a, int n, int first_size, int nseq, int gap, int t) {
  const int nb = __ffs(n) - 1;  // log2(n)
  for (int size = first_size; size <= n; size <<= 1) {
    for (int hi = size >> 1; hi >= 1;) {
      const int ns = hi >= 4 ? 3 : (hi >= 2 ? 2 : 1);
      const int lo = hi >> (ns - 1);
      const int lob = __ffs(lo) - 1;
      const int per_seq = n >> ns;
      const int groups = per_seq * nseq;
      for (int gi = t; gi < groups; gi += T::size) {
        const int q = gi >> (nb - ns);
        const int gl = gi & (per_seq - 1);
        const int base = ((gl >> lob) << (lob + ns)) | (gl & (lo - 1));
        const bool larger_first = ((base & size) == 0) == DESC;
        K* aq = a + q * gap;
        if (ns == 3) bitonic_group<3>(aq, base, lo, larger_first);
        else if (ns == 2) bitonic_group<2>(aq, base, lo, larger_first);
        else bitonic_group<1>(aq, base, lo, larger_first);
      }
      T::sync();
      hi = lo >> 1;
    }
  }
}

}  // namespace topk
