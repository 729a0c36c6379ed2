// Device building blocks for the fused sample · filter · capture kernel (sm_103a).
//
// Everything here works on one CTA's shared memory: order-preserving keys, the counter-based
// Philox generator for the exponential race, deterministic block reductions and scans, a radix
// select of the k-th largest key, a stable in-place compaction and a bitonic sort of 64-bit
// composite keys. None of it depends on the rest of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

namespace sfc {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr uint32_t kKeyLowestFinite = 0x00800000u;  // key of the most negative finite value

// ------------------------------------------------------------------------------------------
// Element types. Logits arrive as bf16 bit patterns or float32; both widen exactly to float.
// ------------------------------------------------------------------------------------------
template <int DT>
struct Elem;

template <>
struct Elem<0> {  // bfloat16
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;  // elements per 16-byte vector
  __device__ __forceinline__ static float load1(const unsigned char* row, int64_t i) {
    const uint32_t b = reinterpret_cast<const uint16_t*>(row)[i];
    return __uint_as_float(b << 16);
  }
  __device__ __forceinline__ static uint32_t word(const uint4& v, int w) {
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
  }
  // Element e of a vector (e is a compile-time constant after unrolling).
  __device__ __forceinline__ static float get(const uint4& v, int e) {
    const uint32_t w = word(v, e >> 1);
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  // Element e of a vector for a runtime e (selects, no dynamic register indexing).
  __device__ __forceinline__ static float get_dyn(const uint4& v, int e) {
    const int w = e >> 1;
    const uint32_t x = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
    return __uint_as_float((e & 1) ? (x & 0xFFFF0000u) : (x << 16));
  }
  // Bit e set when element e is >= t (t a bf16 value), by packed bf16x2 compares.
  __device__ __forceinline__ static uint32_t ge_mask(const uint4& v, float t) {
    const __nv_bfloat162 tt = __float2bfloat162_rn(t);  // exact: t is a bf16 value
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t h = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[i]), tt);  // 0xFFFF per true half
      m |= ((h & 1u) | ((h >> 15) & 2u)) << (2 * i);
    }
    return m;
  }
  // Largest of the 8 values, with packed bf16x2 maxima.
  __device__ __forceinline__ static float vmax(const uint4& v) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                                     *reinterpret_cast<const __nv_bfloat162*>(&v.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                                     *reinterpret_cast<const __nv_bfloat162*>(&v.w));
    const __nv_bfloat162 c = __hmax2(a, b);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(&c);
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  __device__ __forceinline__ static uint4 neg_inf_vec() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&x)[8]) {
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    x[4] = __uint_as_float(v.z << 16);
    x[5] = __uint_as_float(v.z & 0xFFFF0000u);
    x[6] = __uint_as_float(v.w << 16);
    x[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
};

template <>
struct Elem<1> {  // float32
  static constexpr int kBytes = 4;
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load1(const unsigned char* row, int64_t i) {
    return reinterpret_cast<const float*>(row)[i];
  }
  __device__ __forceinline__ static float get(const uint4& v, int e) {
    return __uint_as_float(e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w)));
  }
  __device__ __forceinline__ static float vmax(const uint4& v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  __device__ __forceinline__ static float get_dyn(const uint4& v, int e) {
    return __uint_as_float(e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w)));
  }
  __device__ __forceinline__ static uint4 neg_inf_vec() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
  __device__ __forceinline__ static uint32_t ge_mask(const uint4& v, float t) {
    return static_cast<uint32_t>(__uint_as_float(v.x) >= t) | (static_cast<uint32_t>(__uint_as_float(v.y) >= t) << 1) |
           (static_cast<uint32_t>(__uint_as_float(v.z) >= t) << 2) | (static_cast<uint32_t>(__uint_as_float(v.w) >= t) << 3);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};

// ------------------------------------------------------------------------------------------
// Order-preserving 32-bit keys. Equal logits (with -0 == +0) get equal keys; a larger logit gets
// a larger key. For bf16 inputs the key is the 16-bit key in the high half, low half zero, so a
// key is always the exact key of some element value and key -> value is exact.
// ------------------------------------------------------------------------------------------
template <int DT>
struct Keys;

template <>
struct Keys<0> {
  static constexpr int kDigitPasses = 2;  // 8-bit digits over bits 31..16
  __device__ __forceinline__ static uint32_t key(float x) {
    uint32_t b = __float_as_uint(x) >> 16;
    if (b == 0x8000u) b = 0u;
    const uint32_t k = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
    return k << 16;
  }
  __device__ __forceinline__ static float value(uint32_t k32) {
    const uint32_t k = k32 >> 16;
    const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(b << 16);
  }
};

template <>
struct Keys<1> {
  static constexpr int kDigitPasses = 4;  // 8-bit digits over bits 31..0
  __device__ __forceinline__ static uint32_t key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
};

// Composite key: logit key in the high word, ~id in the low word. Sorting composites in
// descending order gives the canonical support order (logit descending, id ascending).
__device__ __forceinline__ uint64_t make_ckey(uint32_t key, uint32_t id) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~id);
}
__device__ __forceinline__ uint32_t ckey_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ uint32_t ckey_id(uint64_t c) { return ~static_cast<uint32_t>(c); }

// ------------------------------------------------------------------------------------------
// Arithmetic primitives
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {  // 2^x on the SFU; -inf -> +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed f32x2 arithmetic (two float32 lanes in a 64-bit register; sm_100 and later).
__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack_f2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd_f2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {  // max that propagates NaN
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {  // read-once 16-byte load
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// The same load issued exactly once where written: a volatile asm is never re-issued by the
// compiler, so a value held across a long stretch of code stays in registers instead of being
// loaded again from memory.
__device__ __forceinline__ uint4 ld_once(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ------------------------------------------------------------------------------------------
// Bulk asynchronous copies (global -> shared) completing on an mbarrier. Every wait is bounded:
// each poll suspends the thread for at most kWaitSuspendNs, and the wait gives up after
// kWaitPolls polls (a few seconds) and reports it, so a lost completion cannot hang the GPU.
// ------------------------------------------------------------------------------------------
constexpr uint32_t kWaitPolls = 1u << 21;
constexpr uint32_t kWaitSuspendNs = 2000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// Wait for the phase with the given parity to complete; false if it did not within `polls` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t polls = kWaitPolls) {
  const uint32_t a = smem_addr(bar);
  for (uint32_t i = 0; i < polls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity), "n"(kWaitSuspendNs)
        : "memory");
    if (done) return true;
  }
  return false;
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) into this CTA's shared memory;
// the transfer counts against `bar`'s expected transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// ------------------------------------------------------------------------------------------
// Thread-block clusters: a barrier over the cluster's CTAs (release / acquire), and loads from a
// peer CTA's shared memory (distributed shared memory) at the address of a local variable.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint64_t dsmem_ld64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_ld32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}


// Philox4x32-10 (Salmon et al., SC'11, section 4): counter (c0..c3), key (k0, k1); word 0 of
// the output block. Ten rounds: multiply words 0 and 2 by the two round multipliers, swap the
// product halves into the counter XOR-ed with the other words and the round key, bump the key
// by the two Weyl increments.
__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

// Race variate for token `id` of `row` at decode `step`: u in (0,1), exact in float32.
__device__ __forceinline__ float race_uniform(uint64_t seed, uint64_t step, uint32_t row, uint32_t id) {
  const uint32_t w = philox_word0(id, row, static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32),
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(2u * (w >> 9) + 1u) * 0x1p-24f;
}

// Race score of a support member: z - z_max - ln(E), E = -ln(u). Accurate logs: u near 1 gives a
// tiny E whose logarithm decides the winner.
__device__ __forceinline__ float race_score(float zrel, float u) { return zrel - logf(-logf(u)); }

// (score, id) order of the race: larger score wins, equal scores go to the lower id.
__device__ __forceinline__ bool race_better(float s1, uint32_t id1, float s2, uint32_t id2) {
  return (s1 > s2) || (s1 == s2 && id1 < id2);
}

// ------------------------------------------------------------------------------------------
// Barriers over the NT threads of a CTA that work on its row: a named barrier (1) with an explicit
// thread count, so that a CTA may hold one more warp that takes no part in them. With NT the CTA's
// size they are the CTA-wide barrier.
// ------------------------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ void cta_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
// The same barrier, returning whether pred held in any of the NT threads.
template <int NT>
__device__ __forceinline__ bool cta_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(NT)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------------------------------
// Warp / block reductions (fixed combination order, hence deterministic)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_incl_scan_f(float v) {  // fixed order: deterministic
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

template <int NT>
struct Block {
  static constexpr int kWarps = NT / 32;

  // Sum of one float per thread: warp butterflies, then warps in order. Result in every thread.
  __device__ static float sum(float v, float* scratch) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5;
    cta_sync<NT>();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    cta_sync<NT>();
    float t = 0.f;
    for (int i = 0; i < kWarps; ++i) t += scratch[i];
    return t;
  }

  __device__ static int sum_int(int v, int* scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    const int w = threadIdx.x >> 5;
    cta_sync<NT>();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    cta_sync<NT>();
    int t = 0;
    for (int i = 0; i < kWarps; ++i) t += scratch[i];
    return t;
  }

  __device__ static int min_int(int v, int* scratch) {
    v = warp_min_int(v);
    const int w = threadIdx.x >> 5;
    cta_sync<NT>();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    cta_sync<NT>();
    int t = scratch[0];
    for (int i = 1; i < kWarps; ++i) t = min(t, scratch[i]);
    return t;
  }

  // Exclusive prefix of one float per thread (thread order); total returned through `total`.
  __device__ static float excl_scan(float v, float* scratch, float& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    cta_sync<NT>();
    if (lane == 31) scratch[w] = incl;
    cta_sync<NT>();
    float off = 0.f, tot = 0.f;
    for (int i = 0; i < kWarps; ++i) {
      if (i < w) off += scratch[i];
      tot += scratch[i];
    }
    total = tot;
    return off + incl - v;
  }

  // Exclusive prefix of one int per thread (thread order); total returned through `total`.
  __device__ static int excl_scan_int(int v, int* scratch, int& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int incl = warp_incl_scan(v);
    cta_sync<NT>();
    if (lane == 31) scratch[w] = incl;
    cta_sync<NT>();
    int off = 0, tot = 0;
    for (int i = 0; i < kWarps; ++i) {
      if (i < w) off += scratch[i];
      tot += scratch[i];
    }
    total = tot;
    return off + incl - v;
  }

  // Exclusive prefixes of an (int, float) pair per thread in one pass (thread order); totals
  // returned through ti and tf.
  __device__ static void excl_scan2(int& vi, float& vf, int* si, float* sf, int& ti, float& tf) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int ii = vi;
    float ff = vf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(kFull, ii, o);
      const float b = __shfl_up_sync(kFull, ff, o);
      if (lane >= o) {
        ii += a;
        ff += b;
      }
    }
    cta_sync<NT>();
    if (lane == 31) {
      si[w] = ii;
      sf[w] = ff;
    }
    cta_sync<NT>();
    int oi = 0, toti = 0;
    float of = 0.f, totf = 0.f;
    for (int i = 0; i < kWarps; ++i) {
      if (i < w) {
        oi += si[i];
        of += sf[i];
      }
      toti += si[i];
      totf += sf[i];
    }
    ti = toti;
    tf = totf;
    vi = oi + ii - vi;
    vf = of + ff - vf;
  }

  // Minimum / maximum of one float per thread (NaN-ignoring). Result in every thread.
  __device__ static float min_f(float v, float* scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    const int w = threadIdx.x >> 5;
    cta_sync<NT>();
    if ((threadIdx.x & 31) == 0) scratch[w] = v;
    cta_sync<NT>();
    float t = scratch[0];
    for (int i = 1; i < kWarps; ++i) t = fminf(t, scratch[i]);
    return t;
  }

  // Race argmax: best (score, id) over the block; the winner's logit travels with it.
  __device__ static void race_argmax(float& s, uint32_t& id, float& x, float* fs, uint32_t* ids, float* xs) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float s2 = __shfl_xor_sync(kFull, s, o);
      const uint32_t i2 = __shfl_xor_sync(kFull, id, o);
      const float x2 = __shfl_xor_sync(kFull, x, o);
      if (race_better(s2, i2, s, id)) { s = s2; id = i2; x = x2; }
    }
    const int w = threadIdx.x >> 5;
    cta_sync<NT>();
    if ((threadIdx.x & 31) == 0) { fs[w] = s; ids[w] = id; xs[w] = x; }
    cta_sync<NT>();
    s = fs[0]; id = ids[0]; x = xs[0];
    for (int i = 1; i < kWarps; ++i)
      if (race_better(fs[i], ids[i], s, id)) { s = fs[i]; id = ids[i]; x = xs[i]; }
  }
};

// Online softmax statistics: (m, s) means s = sum 2^((x - m) c). Merge two partial states.
__device__ __forceinline__ void stat_merge(float& m, float& s, float m2, float s2, float c) {
  const float mn = fmax_nan(m, m2);
  if (!(mn > -INFINITY)) {  // both empty (or NaN: the row is rejected later)
    m = mn;
    s = 0.f;
    return;
  }
  const float a = (m > -INFINITY) ? s * ex2_approx((m - mn) * c) : 0.f;
  const float b = (m2 > -INFINITY) ? s2 * ex2_approx((m2 - mn) * c) : 0.f;
  m = mn;
  s = a + b;
}

// ------------------------------------------------------------------------------------------
// Shared-memory scratch used by the block algorithms below.
// ------------------------------------------------------------------------------------------
template <int NT>
struct BlockScratch {
  uint32_t* whist;  // [NT / 32][256] warp-private digit histograms (no cross-warp atomic traffic),
                    // in dynamic shared memory: only the sorting and multi-pass finishes use them
  uint32_t hist[256];
  int warp_cnt[NT / 32];
  float red_f[NT / 32];
  int red_i[NT / 32];
  uint32_t red_u[NT / 32];
  float red_x[NT / 32];
  uint32_t sel_prefix;
  int sel_rem;
};

// Block-wide radix select: the exact `rank`-th largest (1-based) key among the high words of
// cand[0..n). Requires 1 <= rank <= n and NT >= 256. Keys are scanned 8 bits at a time from bit 31
// down, for `passes` digits (2 for bf16 keys, 4 for float keys); each pass builds one digit
// histogram per warp, sums them per bin and lets one warp locate the bin holding the rank.
template <int NT>
__device__ __noinline__ uint32_t block_select_key(const uint64_t* cand, int n, int rank, int passes,
                                                  BlockScratch<NT>& sc) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0;
  int rem = rank;
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = lane; i < 256; i += 32) sc.whist[warp * 256 + i] = 0;
    __syncwarp();
    for (int i = tid; i < n; i += NT) {
      const uint32_t key = ckey_key(cand[i]);
      if (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8)))
        atomicAdd(&sc.whist[warp * 256 + ((key >> shift) & 0xFFu)], 1u);
    }
    cta_sync<NT>();
    if (tid < 256) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += sc.whist[w * 256 + tid];
      sc.hist[tid] = t;
    }
    cta_sync<NT>();
    if (warp == 0) {
      int local[8];
      int lsum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        local[j] = static_cast<int>(sc.hist[255 - 8 * lane - j]);
        lsum += local[j];
      }
      const int incl = warp_incl_scan(lsum);
      const int excl = incl - lsum;
      if (excl < rem && rem <= incl) {
        int c = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (c + local[j] >= rem && c < rem) {
            sc.sel_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
            sc.sel_rem = rem - c;
          }
          c += local[j];
        }
      }
    }
    cta_sync<NT>();
    prefix = sc.sel_prefix;
    rem = sc.sel_rem;
  }
  return prefix;
}

// Radix select over keys held in registers (NK per thread, NT threads): the exact `rank`-th
// largest (1-based, rank <= NT*NK) of the NT*NK keys. Same digit scheme as block_select_key.
template <int NT, int NK>
__device__ __forceinline__ uint32_t block_select_regs(const uint32_t (&keys)[NK], int rank, int passes,
                                                      BlockScratch<NT>& sc) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0;
  int rem = rank;
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = lane; i < 256; i += 32) sc.whist[warp * 256 + i] = 0;
    __syncwarp();
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      const uint32_t key = keys[j];
      if (pass == 0 || (key >> (shift + 8)) == (prefix >> (shift + 8)))
        atomicAdd(&sc.whist[warp * 256 + ((key >> shift) & 0xFFu)], 1u);
    }
    cta_sync<NT>();
    if (tid < 256) {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += sc.whist[w * 256 + tid];
      sc.hist[tid] = t;
    }
    cta_sync<NT>();
    if (warp == 0) {
      int local[8];
      int lsum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        local[j] = static_cast<int>(sc.hist[255 - 8 * lane - j]);
        lsum += local[j];
      }
      const int incl = warp_incl_scan(lsum);
      const int excl = incl - lsum;
      if (excl < rem && rem <= incl) {
        int c = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (c + local[j] >= rem && c < rem) {
            sc.sel_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - j) << shift);
            sc.sel_rem = rem - c;
          }
          c += local[j];
        }
      }
    }
    cta_sync<NT>();
    prefix = sc.sel_prefix;
    rem = sc.sel_rem;
  }
  return prefix;
}

// Stable in-place compaction of cand[0..n): keep entries whose key is >= tau. Returns the new
// count (uniform across the block). Chunks of 4*NT entries, 4 consecutive entries per thread: a
// chunk is read completely before any of it is written, and entries only move to lower indices.
template <int NT>
__device__ __noinline__ int block_compact_ge(uint64_t* cand, int n, uint32_t tau, BlockScratch<NT>& sc) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int out = 0;
  for (int base = 0; base < n; base += 4 * NT) {
    uint64_t e[4];
    unsigned keep = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = base + 4 * tid + j;
      e[j] = cand[min(i, n - 1)];  // clamped, unconditional
      keep |= static_cast<unsigned>((i < n) && ckey_key(e[j]) >= tau) << j;
    }
    const int cnt = __popc(keep);
    const int incl = warp_incl_scan(cnt);
    if (lane == 31) sc.warp_cnt[warp] = incl;
    cta_sync<NT>();
    int woff = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int c = sc.warp_cnt[w];
      woff += (w < warp) ? c : 0;
      tot += c;
    }
    int pos = out + woff + incl - cnt;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((keep >> j) & 1) cand[pos++] = e[j];
    out += tot;
    cta_sync<NT>();
  }
  return out;
}

// Bitonic sort of cand[0..n) in place, descending, padded with 0 (which sorts last) up to the
// next power of two P <= capacity. Used only when there is no room for a merge buffer.
template <int NT>
__device__ __noinline__ void block_bitonic_desc(uint64_t* cand, int n) {
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + threadIdx.x; i < P; i += NT) cand[i] = 0ull;
  cta_sync<NT>();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (P >> 1); t += NT) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = cand[lo], b = cand[hi];
        if ((a < b) == desc) {
          cand[lo] = b;
          cand[hi] = a;
        }
      }
      cta_sync<NT>();
    }
  }
}

template <int E>
__device__ __forceinline__ void reg_sort_desc(uint64_t (&v)[E]) {  // bitonic network in registers
#pragma unroll
  for (int size = 2; size <= E; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const uint64_t a = v[i], b = v[j];
          const bool sw = (a < b) == desc;
          v[i] = sw ? b : a;
          v[j] = sw ? a : b;
        }
      }
    }
  }
}

// Merge sort of cand[0..n) descending (n <= NT*E, 2*P <= capacity where P is the padded length):
// every thread sorts E consecutive entries in registers, then runs are merged pairwise with a
// merge-path split per thread (E outputs each), ping-ponging between cand[0..P) and cand[P..2P).
// Returns a pointer to the sorted P entries (zeros pad the end).
template <int NT, int E>
__device__ __noinline__ uint64_t* block_merge_sort_desc(uint64_t* cand, int n) {
  int P = E;
  while (P < n) P <<= 1;
  const int tid = threadIdx.x;
  const int nthr = P / E;  // threads that own a run
  uint64_t* src = cand;
  uint64_t* dst = cand + P;
  if (tid < nthr) {
    uint64_t v[E];
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int i = tid * E + j;
      v[j] = cand[min(i, max(n - 1, 0))];
      if (!(i < n)) v[j] = 0ull;
    }
    reg_sort_desc<E>(v);
#pragma unroll
    for (int j = 0; j < E; ++j) src[tid * E + j] = v[j];
  }
  cta_sync<NT>();
  for (int r = E; r < P; r <<= 1) {
    if (tid < nthr) {
      const int o0 = tid * E;
      const int q = o0 / (2 * r);
      const uint64_t* A = src + q * 2 * r;
      const uint64_t* Bv = A + r;
      const int diag = o0 - q * 2 * r;
      int lo = max(0, diag - r), hi = min(diag, r);
      while (lo < hi) {  // number of A entries among the first `diag` outputs (A wins ties)
        const int mid = (lo + hi) >> 1;
        if (A[mid] >= Bv[diag - mid - 1]) lo = mid + 1;
        else hi = mid;
      }
      int i = lo, j = diag - lo;
      uint64_t* out = dst + q * 2 * r + diag;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        const uint64_t a = A[min(i, r - 1)], b = Bv[min(j, r - 1)];  // reads stay inside the two runs
        const bool takeA = (j >= r) || (i < r && a >= b);
        out[k] = takeA ? a : b;
        i += takeA ? 1 : 0;
        j += takeA ? 0 : 1;
      }
    }
    cta_sync<NT>();
    uint64_t* t = src;
    src = dst;
    dst = t;
  }
  return src;
}

// Sort cand[0..n) descending in a buffer of `cap` entries; returns where the sorted run starts.
template <int NT, int E>
__device__ uint64_t* block_sort_desc(uint64_t* cand, int n, int cap) {
  int P = E;
  while (P < n) P <<= 1;
  if (n <= NT * E && 2 * P <= cap) return block_merge_sort_desc<NT, E>(cand, n);
  block_bitonic_desc<NT>(cand, n);
  return cand;
}

}  // namespace sfc
