// Fused sample · filter · capture kernel for one decode step (sm_103a).
//
// Grid: B clusters of `split` CTAs; cluster c handles row c, CTA rank r streams the r-th slice of
// the row. One HBM read of the logits per row element, in 16-byte vectors:
//
//   stream   each CTA keeps online softmax statistics (running max, sum of 2^((x-m)c)) and a
//            shared-memory buffer of candidate (key, id) pairs above a rising threshold tau.
//            When the buffer fills, a radix select finds the slice's k-th largest key, tau rises
//            to it and the buffer is compacted; ties at tau stay. Every token of the row's top-k
//            set K (ties kept) has fewer than k larger logits in its own slice, so it survives.
//   merge    over distributed shared memory: every CTA shares its tau, the largest of them is a
//            lower bound of the row's k-th largest logit, the leader pulls the other CTAs'
//            statistics and candidates into its own buffer.
//   finish   (leader) exact k-th largest key, sort of K by (logit desc, id asc), exclusive scan
//            of the probability mass in that order -> top-p cut at the first tie group whose
//            mass-above exceeds top_p * Z, min-p cut, renormaliser of S, Philox exponential race
//            over S, packed output for capturing rows.
//   general  rows whose candidates do not fit on chip (top_k disabled or very large on a long
//            row, or a tie group larger than the buffer) are finished by the leader with a few
//            more passes over the row: a radix descent that finds the top-k / top-p threshold with
//            integer counts and fixed-point masses, a pass for |S|, its renormaliser and the race,
//            and, for capturing rows with a support larger than the buffer, two count-only
//            descents that pick the first W support members in canonical order.
//
// Method sources, by page title and section: prhub summary of SGLang PR #36630 (实现拆解 2-4,
// 关键源码片段: joint top-k / top-p thresholds, ties kept, keep-sets intersected, support = positive
// weights); "[Sampling] Stream sampling masks as per-request arrays" (Contract; Checks removed
// item 1: packed per-row arrays, OK/OVERFLOW); "vLLM Sampling Mask（Distribution Replay）深入解析"
// (工作原理 Step 1-2: temperature, min-p, top-k/top-p; finite survivors); "topk-subset-sampler"
// (The fix: one top-k candidate subset, exponential race).
#pragma once

#include <cooperative_groups.h>

#include <cstdint>

#include "sfc_device.cuh"

namespace sfc {

namespace cg = cooperative_groups;

constexpr int kMaxSplit = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFixedScale = 1099511627776.0f;  // 2^40: fixed-point scale of probability weights

enum : int { kModeFast = 0, kModeGeneral = 1, kModeBad = 2 };

struct Params {
  const void* logits;
  int64_t row_stride;  // elements
  int64_t V;
  int32_t B;
  int32_t split;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const float* min_p;
  uint64_t seed;
  uint64_t step;
  const uint8_t* capture_rows;
  int32_t W;
  int32_t* tokens;
  int32_t* support_ids;
  float* support_logprobs;
  int32_t* lengths;
  float* selected_logprob;
  int32_t* row_status;
};

template <int NT>
struct Shared {
  BlockScratch<NT> sc;
  unsigned long long mass[256];
  int count;        // candidates held in the buffer
  uint32_t tau;     // candidate threshold (key); entries below it are never kept
  int spilled;      // the buffer could not hold every token above tau
  uint32_t peer_tau[kMaxSplit];
  float peer_m[kMaxSplit], peer_s[kMaxSplit];
  int peer_off[kMaxSplit + 1];
  float stat_m, stat_s;  // this CTA's softmax statistics
  int mode;              // leader's decision for the row
  // leader scratch
  float row_m, row_Z;
  int peer_count[kMaxSplit];
  // finish / general path results
  float zs;
  int n_sel;
  uint32_t d_prefix;
  int d_rem, d_ka, d_pa, d_done;
  unsigned long long d_mass_above, d_thr;
  int d_cnt_above;
  int gather_overflow;
};

// Per-row constants, identical in every thread of the cluster.
struct RowCtx {
  int row;
  int64_t V;
  float T, c, top_p, ln_min_p;
  int k;
  bool k_active, p_active, m_active, capture;
  const unsigned char* rowp;
  int64_t head, nvec, body_end;
};

__device__ __forceinline__ float zrel_of(float x, float m, float T) { return (x - m) / T; }

__device__ __forceinline__ void write_bad_row(const Params& p, int row, bool capture) {
  p.tokens[row] = -1;
  p.row_status[row] = -1;
  if (p.lengths) p.lengths[row] = 0;
  if (capture && p.selected_logprob) p.selected_logprob[row] = __int_as_float(0x7FC00000);
}

// Visit every element of the row once: unaligned head, 16-byte vectors, ragged tail. Every thread
// runs the same number of rounds and calls f(x, id, valid) in each (invalid lanes carry a clamped
// copy of a real element), so f may use warp collectives. Each thread sees the same elements in
// the same order on every pass, so per-thread sums are deterministic.
template <int DT, int NT, typename F>
__device__ __forceinline__ void row_pass(const RowCtx& rc, F&& f) {
  using E = Elem<DT>;
  constexpr int VEC = E::kVec;
  const int tid = threadIdx.x;
  if (rc.head > 0) {  // uniform; head < VEC <= NT
    const bool v = tid < rc.head;
    f(E::load1(rc.rowp, v ? tid : 0), static_cast<uint32_t>(tid), v);
  }
  const uint4* vb = reinterpret_cast<const uint4*>(rc.rowp + rc.head * E::kBytes);
  const int64_t rounds = (rc.nvec + NT - 1) / NT;
  for (int64_t r = 0; r < rounds; ++r) {
    const int64_t j = r * NT + tid;
    const bool v = j < rc.nvec;
    const uint4 w = ld_stream(vb + min(j, rc.nvec - 1));
    const uint32_t id0 = static_cast<uint32_t>(rc.head + j * VEC);
#pragma unroll
    for (int e = 0; e < VEC; ++e) f(E::get(w, e), id0 + e, v);
  }
  if (rc.body_end < rc.V) {  // uniform; tail < VEC <= NT
    const int64_t i = rc.body_end + tid;
    const bool v = i < rc.V;
    f(E::load1(rc.rowp, v ? i : rc.V - 1), static_cast<uint32_t>(i), v);
  }
}

// Warp-aggregated histogram increment: lanes with equal digits add once (by their lowest lane).
// All 32 lanes must call it; lanes with valid == false add nothing.
__device__ __forceinline__ void warp_hist_inc(uint32_t* hist, uint32_t d, bool valid) {
  const unsigned same = __match_any_sync(kFull, valid ? d : 0xFFFFFFFFu);
  if (valid && static_cast<int>(threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[d], static_cast<uint32_t>(__popc(same)));
}

// Warp-aggregated append of one entry per lane (lanes with take == false append nothing) at
// cand[*count ...]; entries at or past `cap` are counted but not written. All lanes must call it.
__device__ __forceinline__ void warp_append(uint64_t* cand, int* count, int cap, uint64_t e, bool take) {
  const int lane = threadIdx.x & 31;
  const unsigned b = __ballot_sync(kFull, take);
  int base = 0;
  if (lane == 0 && b) base = atomicAdd(count, __popc(b));
  base = __shfl_sync(kFull, base, 0);
  const int pos = base + __popc(b & ((1u << lane) - 1u));
  if (take && pos < cap) cand[pos] = e;
}

// ------------------------------------------------------------------------------------------
// Streaming state of one CTA.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int BUF, int U>
struct Streamer {
  using K = Keys<DT>;
  using E = Elem<DT>;
  static constexpr int VEC = E::kVec;
  static constexpr int SV = 2;  // sample vectors per thread for the threshold estimate
  uint64_t* cand;
  Shared<NT>& sh;
  // row constants, copied (the streaming loop keeps them in registers)
  struct {
    float c;
    int k;
    bool k_active;
    const unsigned char* rowp;
    int64_t head;
  } rc;
  float m_t = -INFINITY, s_t = 0.f;  // online softmax state of this thread
  uint32_t tau = kKeyLowestFinite;   // candidate threshold (key) and its value
  float tau_f;
  uint4 cur[U];                       // the current tile, in registers
  uint32_t id_t0;                     // id of element 0 of this thread's vector 0 in the tile
  float xe;                           // one extra scalar (unaligned head / ragged tail), -inf if none
  uint32_t ide;

  __device__ Streamer(uint64_t* c, Shared<NT>& s, const RowCtx& r) : cand(c), sh(s) {
    rc.c = r.c;
    rc.k = r.k;
    rc.k_active = r.k_active;
    rc.rowp = r.rowp;
    rc.head = r.head;
    tau_f = K::value(tau);
  }

  __device__ __forceinline__ float tile_max() const {
    float m = xe;
#pragma unroll
    for (int u = 0; u < U; ++u) m = fmaxf(m, E::vmax(cur[u]));
    return m;
  }

  // Fold the tile into the statistics. NaN and +inf are not tested element by element: +inf
  // becomes the maximum and NaN poisons the sum, and the row is rejected from either. The tile's
  // partial sum (a short tree per thread) keeps the per-thread total accurate without Kahan steps.
  __device__ __forceinline__ void absorb(float tmax) {
    if (!(tmax <= m_t)) {
      const float mn = fmaxf(m_t, tmax);
      if (m_t > -INFINITY) s_t *= ex2_approx((m_t - mn) * rc.c);
      m_t = mn;
    }
    const float nmc = -fmaxf(m_t, -FLT_MAX) * rc.c;  // 2^(x c - m c); -inf lanes give 0
    float a0 = ex2_approx(fmaf(xe, rc.c, nmc)), a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int e = 0; e < VEC; e += 2) {
        float& acc = (u & 1) ? a2 : a0;
        float& acd = (u & 1) ? a3 : a1;
        acc += ex2_approx(fmaf(E::get(cur[u], e), rc.c, nmc));
        acd += ex2_approx(fmaf(E::get(cur[u], e + 1), rc.c, nmc));
      }
    }
    s_t += (a0 + a1) + (a2 + a3);
  }

  // Append this thread's tile elements >= tau_f (and the extra scalar). Per-thread shared atomic;
  // no warp collective, so the divergent call is safe. Entries that would pass the end of the
  // buffer are not written and flag the row for the multi-pass path.
  __device__ __forceinline__ void append() {
    uint64_t take = 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int e = 0; e < VEC; ++e) take |= static_cast<uint64_t>(E::get(cur[u], e) >= tau_f) << (8 * u + e);
    }
    take |= static_cast<uint64_t>(xe >= tau_f) << (8 * U);
    const int cnt = __popcll(take);
    if (cnt == 0) return;
    int pos = atomicAdd(&sh.count, cnt);
    if (pos + cnt > BUF) sh.spilled = 1;
    while (take) {
      const int bit = __ffsll(static_cast<long long>(take)) - 1;
      take &= take - 1;
      float x;
      uint32_t id;
      if (bit == 8 * U) {
        x = xe;
        id = ide;
      } else {
        const int u = bit >> 3, e = bit & 7;
        uint4 v = cur[0];
#pragma unroll
        for (int q = 1; q < U; ++q) v = (u == q) ? cur[q] : v;
        x = E::get_dyn(v, e);
        id = id_t0 + static_cast<uint32_t>(u * NT * VEC + e);
      }
      if (pos < BUF) cand[pos] = make_ckey(K::key(x), id);
      ++pos;
    }
  }

  // Threshold estimate from an evenly strided sample of the slice (SV vectors per thread, plus the
  // extra scalars). With a sample fraction f, the ks-th largest sample value (ks a high quantile of
  // the number of sampled elements among the slice's k largest) is a lower bound of the slice's
  // (hence the row's) k-th largest logit with overwhelming probability, and the finish verifies
  // that it was one. When the sample is the whole slice, ks = k and the bound is exact.
  __device__ void sample_threshold(const uint4* sb, int nvec, int n_extra) {
    if (!rc.k_active) return;
    constexpr int NK = SV * VEC + 1;
    const int ns = min(SV * NT, nvec);
    uint32_t keys[NK];
#pragma unroll
    for (int q = 0; q < SV; ++q) {
      const int i = q * NT + static_cast<int>(threadIdx.x);
      const bool valid = i < ns;
      const int j = (ns == nvec) ? i : static_cast<int>((static_cast<int64_t>(i) * nvec) / max(ns, 1));
      const uint4 v = nvec > 0 ? ld_stream(sb + min(j, max(nvec - 1, 0))) : E::neg_inf_vec();
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float x = E::get(v, e);
        keys[q * VEC + e] = (valid && x > -INFINITY && x < INFINITY) ? K::key(x) : 0u;
      }
    }
    keys[NK - 1] = (xe > -INFINITY && xe < INFINITY) ? K::key(xe) : 0u;
    const bool whole = ns == nvec;
    const int64_t slice = static_cast<int64_t>(nvec) * VEC + n_extra;
    const int64_t sampled = static_cast<int64_t>(ns) * VEC + n_extra;
    int ks;
    if (whole) {
      ks = rc.k;
    } else {
      // The number of sampled elements among the slice's k-1 largest is about Poisson(lam),
      // lam = (k-1) f. The estimate fails only if at least ks of them were sampled; with
      // ks = lam + 5.3 sqrt(lam) + 6 that has probability below about 1e-7.
      const float lam = static_cast<float>(rc.k) * static_cast<float>(sampled) / static_cast<float>(slice);
      ks = static_cast<int>(ceilf(lam + 5.3f * sqrtf(lam) + 6.f));
    }
    if (ks > NK * NT) return;  // the sample cannot bound it: no filtering
    const uint32_t t = block_select_regs<NT, NK>(keys, ks, K::kDigitPasses, sh.sc);
    tau = max(t, kKeyLowestFinite);
    tau_f = K::value(tau);
    if (threadIdx.x == 0) sh.tau = tau;
  }

  // One pass over the slice: vectors [vbeg, vend) of the row body, plus `n_head` unaligned
  // leading elements and the `n_tail` elements from `tail_beg`, handed out one per thread and
  // folded into the first tile. No barrier inside the loop: warps run independently.
  __device__ void stream(int64_t vbeg, int64_t vend, int n_head, int64_t tail_beg, int n_tail) {
    const int tid = threadIdx.x;
    const uint4* vb = reinterpret_cast<const uint4*>(rc.rowp + rc.head * E::kBytes);
    const int n_extra = n_head + n_tail;
    xe = -INFINITY;
    ide = 0;
    if (n_extra > 0) {  // uniform; the load is clamped to a valid index and masked by a select
      const bool has = tid < n_extra;
      const int64_t idx = !has ? (n_head > 0 ? 0 : tail_beg) : (tid < n_head ? tid : tail_beg + (tid - n_head));
      const float v = E::load1(rc.rowp, idx);
      xe = has ? v : -INFINITY;
      ide = static_cast<uint32_t>(idx);
    }
    const uint4* sb = vb + vbeg;
    const int nvec = static_cast<int>(vend - vbeg);
    sample_threshold(sb, nvec, n_extra);
    const int ntiles = max((nvec + U * NT - 1) / (U * NT), static_cast<int>(n_extra > 0));
    const int vlast = nvec > 0 ? nvec - 1 : 0;
    const uint32_t id_base = static_cast<uint32_t>(rc.head + vbeg * VEC);
    for (int t = 0; t < ntiles; ++t) {
      const int t0 = t * (U * NT);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = t0 + u * NT + tid;
        cur[u] = nvec > 0 ? ld_stream(sb + min(j, vlast)) : E::neg_inf_vec();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = t0 + u * NT + tid;
        if (!(j < nvec)) cur[u] = E::neg_inf_vec();  // select, not a branch around a load
      }
      id_t0 = id_base + static_cast<uint32_t>(t0 + tid) * VEC;
      const float tmax = tile_max();
      absorb(tmax);
      if (tmax >= tau_f) append();
      xe = -INFINITY;  // the extra element belongs to the first tile only
    }
  }

  // Block-wide: raise tau to the k-th largest buffered key and drop what is below. If that
  // cannot bring the buffer under `limit` (top-k disabled, or ties), give up on candidates.
  __device__ void compact(int limit) {
    const int n = min(sh.count, BUF);
    if (rc.k_active && n > rc.k) {
      const uint32_t t = block_select_key<NT>(cand, n, rc.k, K::kDigitPasses, sh.sc);
      const int nk = block_compact_ge<NT>(cand, n, t, sh.sc);
      if (threadIdx.x == 0) {
        sh.count = nk;
        sh.tau = max(sh.tau, t);
        if (nk > limit) sh.spilled = 1;
      }
    } else {
      __syncthreads();
      if (threadIdx.x == 0) {
        sh.count = n;
        sh.spilled = 1;
      }
    }
    __syncthreads();
    tau = sh.tau;
    tau_f = K::value(tau);
  }

  // Leader: pull the other CTAs' candidates (distributed shared memory) through the filter
  // key >= tau, all peers as one concatenated list, one entry per thread per round.
  __device__ void merge_peers(cg::cluster_group& cluster, int s) {
    constexpr int TRIGGER = BUF - NT;
    const int lane = threadIdx.x & 31;
    const int total = sh.peer_off[s];
    // A round appends at most NT entries: start every round at or below BUF - NT.
    if (total > 0 && !sh.spilled && sh.count > TRIGGER) compact(TRIGGER);
    for (int base = 0; base < total; base += NT) {
      const bool spilled = sh.spilled != 0;  // uniform: read after the previous round's barrier
      const int i = min(base + static_cast<int>(threadIdx.x), total - 1);  // clamped, unconditional
      int r = 1;  // peer holding entry i: count the peer boundaries at or below i (no data-dependent loop)
#pragma unroll
      for (int q = 2; q < kMaxSplit; ++q) r += (q < s && sh.peer_off[q] <= i) ? 1 : 0;
      const uint64_t* peer = cluster.map_shared_rank(cand, r);
      const uint64_t e = peer[i - sh.peer_off[r]];
      const bool take = (base + static_cast<int>(threadIdx.x) < total) && !spilled && ckey_key(e) >= tau;
      bool crossed = false;
      const unsigned b = __ballot_sync(kFull, take);
      if (b) {
        int pos = 0;
        if (lane == 0) {
          pos = atomicAdd(&sh.count, __popc(b));
          crossed = pos + __popc(b) > TRIGGER;
        }
        pos = __shfl_sync(kFull, pos, 0);
        const int dst = pos + __popc(b & ((1u << lane) - 1u));
        if (take) {
          if (dst < BUF) cand[dst] = e;
          else sh.spilled = 1;  // cannot happen (fill <= BUF - NT per round); the row would go multi-pass
        }
      }
      if (__syncthreads_or(crossed)) compact(TRIGGER);
      __syncthreads();
    }
  }
};

// ------------------------------------------------------------------------------------------
// Leader finish when every candidate is on chip: cand[0..n) holds all tokens >= some tau that
// is <= the row's k-th largest logit (or every finite token when top-k is off).
// Returns false (nothing written) if K does not fit the sort buffer.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int BUF>
__device__ __noinline__ bool finish_fast(const Params& p, const RowCtx rc, uint64_t* cand, Shared<NT>& sh, int n,
                                         float m, float Z, uint32_t tau_floor) {
  using K = Keys<DT>;
  constexpr int SORT_E = (NT >= 512) ? 16 : 8;  // register-sorted run length of the merge sort
  constexpr int SORT_CAP = (BUF & (BUF - 1)) == 0 ? BUF : (1 << (31 - __builtin_clz(BUF)));
  const int tid = threadIdx.x;
  // The buffer holds every row element >= tau_floor (each slice kept all its elements above its
  // own threshold, and tau_floor is at least the largest of those). If the buffer's k-th largest
  // is >= tau_floor, the top-k with ties is complete; otherwise some slice's estimate was too high
  // and the multi-pass path takes the row.
  if (rc.k_active) {
    if (n > rc.k) {
      const uint32_t t = block_select_key<NT>(cand, n, rc.k, K::kDigitPasses, sh.sc);
      if (t < tau_floor) return false;
      n = block_compact_ge<NT>(cand, n, t, sh.sc);
    } else if (tau_floor > kKeyLowestFinite) {
      return false;
    }
  }
  if (n < 1 || n > SORT_CAP) return false;
  cand = block_sort_desc<NT, SORT_E>(cand, n, BUF);

  // Exclusive scan of the weights 2^((x-m)c) in canonical order; cut at the first tie group
  // whose mass above exceeds top_p * Z, or whose z - z_max falls below ln(min_p).
  const int C = (n + NT - 1) / NT;
  const int i0 = min(tid * C, n), i1 = min(i0 + C, n);
  float part = 0.f;
  for (int i = i0; i < i1; ++i) part += ex2_approx((K::value(ckey_key(cand[i])) - m) * rc.c);
  float total;
  const float off = Block<NT>::excl_scan(part, sh.sc.red_f, total);
  const float thr = rc.top_p * Z;
  int cut = n;
  {
    float pre = off;
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = ckey_key(cand[i]);
      const float x = K::value(key);
      const bool gstart = (i == 0) || ckey_key(cand[i - 1]) != key;
      if (gstart && cut == n) {
        if (rc.p_active && pre > thr) cut = i;
        if (rc.m_active && zrel_of(x, m, rc.T) < rc.ln_min_p) cut = i;
      }
      pre += ex2_approx((x - m) * rc.c);
    }
  }
  cut = Block<NT>::min_int(cut, sh.sc.red_i);
  const int nS = cut;  // >= 1: the first group always passes
  if (tid == (nS - 1) / C) {
    float pre = off;
    for (int i = i0; i < nS; ++i) pre += ex2_approx((K::value(ckey_key(cand[i])) - m) * rc.c);
    sh.zs = pre;
  }
  __syncthreads();
  const float logZS = logf(sh.zs);

  // Exponential race over S.
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
  for (int i = tid; i < nS; i += NT) {
    const uint64_t ck = cand[i];
    const float x = K::value(ckey_key(ck));
    const uint32_t id = ckey_id(ck);
    const float sc = race_score(zrel_of(x, m, rc.T), race_uniform(p.seed, p.step, static_cast<uint32_t>(rc.row), id));
    if (race_better(sc, id, best, bid)) { best = sc; bid = id; bx = x; }
  }
  Block<NT>::race_argmax(best, bid, bx, sh.sc.red_f, sh.sc.red_u, sh.sc.red_x);

  if (tid == 0) {
    p.tokens[rc.row] = static_cast<int32_t>(bid);
    if (rc.capture) {
      p.lengths[rc.row] = nS;
      p.row_status[rc.row] = nS > p.W ? 1 : 0;
      p.selected_logprob[rc.row] = zrel_of(bx, m, rc.T) - logZS;
    } else {
      p.row_status[rc.row] = 0;
      if (p.lengths) p.lengths[rc.row] = 0;
    }
  }
  if (rc.capture) {
    const int n_out = min(nS, p.W);
    int32_t* ids = p.support_ids + static_cast<int64_t>(rc.row) * p.W;
    float* lps = p.support_logprobs ? p.support_logprobs + static_cast<int64_t>(rc.row) * p.W : nullptr;
    for (int i = tid; i < n_out; i += NT) {
      const uint64_t ck = cand[i];
      ids[i] = static_cast<int32_t>(ckey_id(ck));
      if (lps) lps[i] = zrel_of(K::value(ckey_key(ck)), m, rc.T) - logZS;
    }
  }
  return true;
}

// ------------------------------------------------------------------------------------------
// General path (leader CTA alone, several passes over the row).
// ------------------------------------------------------------------------------------------

// Count-only radix descent over a per-element 32-bit value among the elements `sel` accepts:
// returns the rank-th largest value and, through cnt_above, how many accepted elements exceed it.
template <int DT, int NT, typename Sel, typename Val>
__device__ uint32_t general_descent_count(const RowCtx& rc, Shared<NT>& sh, int rank, int passes, Sel&& sel,
                                          Val&& val, int& cnt_above) {
  constexpr int kWarps = NT / 32;
  const int warp = threadIdx.x >> 5;
  uint32_t prefix = 0;
  int rem = rank, above = 0;
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < kWarps * 256; i += NT) (&sh.sc.whist[0][0])[i] = 0;
    __syncthreads();
    row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
      bool ok = valid && sel(x, id);
      const uint32_t v = val(x, id);
      if (pass > 0) ok = ok && (v >> (shift + 8)) == (prefix >> (shift + 8));
      warp_hist_inc(sh.sc.whist[warp], (v >> shift) & 0xFFu, ok);
    });
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += NT) {
      uint32_t t = 0;
      for (int w = 0; w < kWarps; ++w) t += sh.sc.whist[w][b];
      sh.sc.hist[b] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, b = 255;
      for (; b > 0; --b) {
        const int cb = static_cast<int>(sh.sc.hist[b]);
        if (cum + cb >= rem) break;
        cum += cb;
      }
      sh.d_prefix = prefix | (static_cast<uint32_t>(b) << shift);
      sh.d_rem = rem - cum;
      sh.d_cnt_above = above + cum;
    }
    __syncthreads();
    prefix = sh.d_prefix;
    rem = sh.d_rem;
    above = sh.d_cnt_above;
    __syncthreads();
  }
  cnt_above = above;
  return prefix;
}

template <int DT, int NT, int BUF>
__device__ __noinline__ void general_path(const Params& p, const RowCtx rc, uint64_t* cand, Shared<NT>& sh, float m,
                                          float Z) {
  using K = Keys<DT>;
  constexpr int SORT_E = (NT >= 512) ? 16 : 8;
  constexpr int kWarps = NT / 32;
  static_assert(BUF >= NT * 8, "the mass histograms borrow the candidate buffer");
  const int warp = threadIdx.x >> 5;
  constexpr int SORT_CAP = (BUF & (BUF - 1)) == 0 ? BUF : (1 << (31 - __builtin_clz(BUF)));
  const int tid = threadIdx.x;
  const float c = rc.c;

  // 1. Threshold tau = max(kcut, pcut): radix descent with integer counts (top-k) and 2^-40
  //    fixed-point weights (top-p), 8 bits of the key per pass.
  if (tid == 0) {
    sh.d_prefix = 0;
    sh.d_rem = rc.k;
    sh.d_ka = rc.k_active;
    sh.d_pa = rc.p_active;
    sh.d_mass_above = 0;
    sh.d_thr = 0;
    sh.d_done = !(rc.k_active || rc.p_active);
  }
  __syncthreads();
  for (int level = 0; level < K::kDigitPasses; ++level) {
    if (sh.d_done) break;
    const int shift = 24 - 8 * level;
    const uint32_t prefix = sh.d_prefix;
    const bool pa = sh.d_pa;
    // Warp-private count and fixed-point mass histograms (the mass ones live in the candidate
    // buffer, unused until the gather); integer sums, so the order of the adds does not matter.
    unsigned long long* wmass = reinterpret_cast<unsigned long long*>(cand);
    for (int i = tid; i < kWarps * 256; i += NT) {
      (&sh.sc.whist[0][0])[i] = 0;
      wmass[i] = 0;
    }
    __syncthreads();
    row_pass<DT, NT>(rc, [&](float x, uint32_t, bool valid) {
      const uint32_t key = K::key(x);
      bool ok = valid && x > -INFINITY;
      if (level > 0) ok = ok && (key >> (shift + 8)) == (prefix >> (shift + 8));
      const uint32_t d = (key >> shift) & 0xFFu;
      warp_hist_inc(sh.sc.whist[warp], d, ok);
      if (pa && ok) atomicAdd(&wmass[warp * 256 + d], static_cast<unsigned long long>(__float2ull_rn(ex2_approx((x - m) * c) * kFixedScale)));
    });
    __syncthreads();
    for (int b = tid; b < 256; b += NT) {
      uint32_t t = 0;
      unsigned long long mm = 0;
      for (int w = 0; w < kWarps; ++w) {
        t += sh.sc.whist[w][b];
        mm += wmass[w * 256 + b];
      }
      sh.sc.hist[b] = t;
      sh.mass[b] = mm;
    }
    __syncthreads();
    if (tid == 0) {
      bool ka = sh.d_ka, pa0 = sh.d_pa;
      int rem = sh.d_rem;
      if (level == 0) {
        int tot = 0;
        unsigned long long mtot = 0;
        for (int b = 0; b < 256; ++b) {
          tot += static_cast<int>(sh.sc.hist[b]);
          mtot += sh.mass[b];
        }
        if (ka && tot <= rc.k) ka = false;  // at most k finite tokens: K is every finite token
        if (pa0) sh.d_thr = static_cast<unsigned long long>(static_cast<double>(rc.top_p) * static_cast<double>(mtot));
      }
      const unsigned long long thr = sh.d_thr;
      int bk = -1, bp = -1;
      if (ka) {
        int cum = 0;
        for (int b = 255; b >= 0; --b) {
          const int cb = static_cast<int>(sh.sc.hist[b]);
          if (cum + cb >= rem) { bk = b; break; }
          cum += cb;
        }
      }
      if (pa0) {
        unsigned long long before = sh.d_mass_above;
        for (int b = 255; b >= 0; --b) {
          if (before > thr) break;
          if (sh.sc.hist[b] > 0) bp = b;
          before += sh.mass[b];
        }
      }
      const int bstar = max(bk, bp);
      if (bstar < 0) {
        sh.d_done = 1;
        sh.d_ka = 0;
        sh.d_pa = 0;
      } else {
        if (ka && bk < bstar) ka = false;
        if (pa0 && bp < bstar) pa0 = false;
        int cnt_above = 0;
        unsigned long long mass_above = 0;
        for (int b = 255; b > bstar; --b) {
          cnt_above += static_cast<int>(sh.sc.hist[b]);
          mass_above += sh.mass[b];
        }
        sh.d_rem = rem - cnt_above;
        sh.d_mass_above += mass_above;
        sh.d_prefix = prefix | (static_cast<uint32_t>(bstar) << shift);
        sh.d_ka = ka;
        sh.d_pa = pa0;
      }
    }
    __syncthreads();
  }
  // With neither constraint ever active the threshold stays 0: every finite token passes.
  const uint32_t tau = sh.d_prefix;
  __syncthreads();

  auto in_S = [&](float x) -> bool {
    if (!(x > -INFINITY)) return false;
    if (K::key(x) < tau) return false;
    if (rc.m_active && zrel_of(x, m, rc.T) < rc.ln_min_p) return false;
    return true;
  };

  // 2. |S|, its renormaliser, the race; gather S when the row captures and S fits.
  if (tid == 0) {
    sh.count = 0;
    sh.gather_overflow = 0;
  }
  __syncthreads();
  int n_loc = 0;
  float zs = 0.f, zc = 0.f;
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
  row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
    const bool ok = valid && in_S(x);
    if (rc.capture) warp_append(cand, &sh.count, SORT_CAP, make_ckey(K::key(x), id), ok);  // collective first
    if (!ok) return;
    ++n_loc;
    const float y = ex2_approx((x - m) * c) - zc;
    const float t = zs + y;
    zc = (t - zs) - y;
    zs = t;
    const float sc = race_score(zrel_of(x, m, rc.T), race_uniform(p.seed, p.step, static_cast<uint32_t>(rc.row), id));
    if (race_better(sc, id, best, bid)) { best = sc; bid = id; bx = x; }
  });
  const float ZS = Block<NT>::sum(zs, sh.sc.red_f);
  const int nS = Block<NT>::sum_int(n_loc, sh.sc.red_i);
  Block<NT>::race_argmax(best, bid, bx, sh.sc.red_f, sh.sc.red_u, sh.sc.red_x);
  const float logZS = logf(ZS);
  if (tid == 0) {
    p.tokens[rc.row] = static_cast<int32_t>(bid);
    if (rc.capture) {
      p.lengths[rc.row] = nS;
      p.row_status[rc.row] = nS > p.W ? 1 : 0;
      p.selected_logprob[rc.row] = zrel_of(bx, m, rc.T) - logZS;
    } else {
      p.row_status[rc.row] = 0;
      if (p.lengths) p.lengths[rc.row] = 0;
    }
  }
  if (!rc.capture) return;
  __syncthreads();

  // 3. The first min(|S|, W) members in canonical order.
  const int n_out = min(nS, p.W);
  if (nS > SORT_CAP) {
    // W-th largest key within S, then the lowest ids among the tokens tied at it.
    int c_gt = 0;
    const uint32_t tW = general_descent_count<DT, NT>(
        rc, sh, n_out, K::kDigitPasses, [&](float x, uint32_t) { return in_S(x); },
        [&](float x, uint32_t) { return K::key(x); }, c_gt);
    int dummy = 0;
    const uint32_t idinvW = general_descent_count<DT, NT>(
        rc, sh, n_out - c_gt, 4, [&](float x, uint32_t) { return in_S(x) && K::key(x) == tW; },
        [&](float, uint32_t id) { return ~id; }, dummy);
    if (tid == 0) sh.count = 0;
    __syncthreads();
    row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
      const uint32_t key = K::key(x);
      const bool ok = valid && in_S(x) && (key > tW || (key == tW && ~id >= idinvW));
      warp_append(cand, &sh.count, SORT_CAP, make_ckey(key, id), ok);
    });
    __syncthreads();
  }
  const int n_have = min(sh.count, SORT_CAP);
  __syncthreads();
  cand = block_sort_desc<NT, SORT_E>(cand, n_have, BUF);
  int32_t* ids = p.support_ids + static_cast<int64_t>(rc.row) * p.W;
  float* lps = p.support_logprobs ? p.support_logprobs + static_cast<int64_t>(rc.row) * p.W : nullptr;
  for (int i = tid; i < n_out; i += NT) {
    const uint64_t ck = cand[i];
    ids[i] = static_cast<int32_t>(ckey_id(ck));
    if (lps) lps[i] = zrel_of(K::value(ckey_key(ck)), m, rc.T) - logZS;
  }
}

// ------------------------------------------------------------------------------------------
// The kernel.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int BUF, int U, int MINB>
__global__ void __launch_bounds__(NT, MINB) fused_kernel(const Params p) {
  using E = Elem<DT>;
  constexpr int VEC = E::kVec;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(dyn_smem);
  __shared__ Shared<NT> sh;

  cg::cluster_group cluster = cg::this_cluster();
  const int s = p.split;
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = static_cast<int>(blockIdx.x) / s;
  const int tid = threadIdx.x;

  RowCtx rc;
  rc.row = row;
  rc.V = p.V;
  rc.T = p.temperature[row];
  rc.k = p.top_k[row];
  rc.top_p = p.top_p[row];
  const float min_p = p.min_p[row];
  rc.capture = p.capture_rows != nullptr && p.capture_rows[row] != 0;
  const bool params_ok = (rc.T > 0.f) && (rc.T < INFINITY) && (rc.top_p >= 0.f) && (min_p >= 0.f) && (min_p <= 1.f);
  if (!params_ok) {  // every CTA of the cluster takes this branch: no cluster barrier is skipped
    if (rank == 0 && tid == 0) write_bad_row(p, row, rc.capture);
    return;
  }
  rc.c = kLog2e / rc.T;
  rc.k_active = rc.k >= 1 && static_cast<int64_t>(rc.k) < rc.V;
  rc.p_active = rc.top_p < 1.f;
  rc.m_active = min_p > 0.f;
  rc.ln_min_p = rc.m_active ? logf(min_p) : -INFINITY;
  rc.rowp = static_cast<const unsigned char*>(p.logits) + static_cast<int64_t>(row) * p.row_stride * E::kBytes;
  rc.head = static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(rc.rowp) & 15u)) & 15u) / E::kBytes;
  if (rc.head > rc.V) rc.head = rc.V;
  rc.nvec = (rc.V - rc.head) / VEC;
  rc.body_end = rc.head + rc.nvec * VEC;

  if (tid == 0) {
    sh.count = 0;
    sh.tau = kKeyLowestFinite;
    sh.spilled = 0;
  }
  __syncthreads();
  // Distributed shared memory may only be touched once every CTA of the cluster is running:
  // arrive now, wait just before the first remote access.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // ---- stream this CTA's slice ----
  Streamer<DT, NT, BUF, U> st(cand, sh, rc);
  const int64_t vbeg = rc.nvec * rank / s, vend = rc.nvec * (rank + 1) / s;
  st.stream(vbeg, vend, rank == 0 ? static_cast<int>(rc.head) : 0, rc.body_end,
            rank == s - 1 ? static_cast<int>(rc.V - rc.body_end) : 0);
  __syncthreads();

  // Block softmax statistics in a fixed order.
  {
    float m = st.m_t, sm = st.s_t;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(kFull, m, o), s2 = __shfl_xor_sync(kFull, sm, o);
      stat_merge(m, sm, m2, s2, rc.c);
    }
    if ((tid & 31) == 0) {
      sh.sc.red_f[tid >> 5] = m;
      sh.sc.red_x[tid >> 5] = sm;
    }
    __syncthreads();
    if (tid == 0) {
      float bm = sh.sc.red_f[0], bs = sh.sc.red_x[0];
      for (int w = 1; w < NT / 32; ++w) stat_merge(bm, bs, sh.sc.red_f[w], sh.sc.red_x[w], rc.c);
      sh.stat_m = bm;
      sh.stat_s = bs;
    }
  }
  __syncthreads();

  // ---- cluster exchange: the leader pulls statistics, thresholds and candidates ----
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster is running
  cluster.sync();  // #1: every CTA's statistics, threshold and candidates are final

  if (rank == 0) {
    if (tid < s) {  // one thread per CTA of the cluster
      const Shared<NT>* peer = cluster.map_shared_rank(&sh, tid);
      sh.peer_m[tid] = peer->stat_m;
      sh.peer_s[tid] = peer->stat_s;
      sh.peer_tau[tid] = peer->tau;
      sh.peer_count[tid] = (peer->spilled || peer->count > BUF) ? -1 : peer->count;
    }
    __syncthreads();
    if (tid == 0) {
      float m = sh.peer_m[0], Z = sh.peer_s[0];
      bool any_spill = sh.peer_count[0] < 0;
      uint32_t lb = sh.peer_tau[0];
      int off = 0;
      for (int r = 1; r < s; ++r) {  // rank order: deterministic
        stat_merge(m, Z, sh.peer_m[r], sh.peer_s[r], rc.c);
        any_spill |= sh.peer_count[r] < 0;
        lb = max(lb, sh.peer_tau[r]);
        sh.peer_off[r] = off;
        off += max(sh.peer_count[r], 0);
      }
      sh.peer_off[s] = off;
      sh.row_m = m;
      sh.row_Z = Z;
      // NaN (poisons the sum), +inf (becomes the maximum) or no finite logit at all.
      const bool bad = !(m > -INFINITY && m < INFINITY) || !(Z == Z);
      sh.mode = bad ? kModeBad : (any_spill ? kModeGeneral : kModeFast);
      // Every CTA's threshold is at most its slice's k-th largest logit, so their maximum is a
      // lower bound of the row's: candidates below it can be dropped.
      sh.tau = max(sh.tau, lb);
    }
    __syncthreads();
    if (sh.mode == kModeFast && s > 1) {
      st.tau = sh.tau;
      st.tau_f = Keys<DT>::value(st.tau);
      st.merge_peers(cluster, s);
      __syncthreads();
      if (tid == 0 && sh.spilled) sh.mode = kModeGeneral;
      __syncthreads();
    }
  }
  cluster.sync();  // #2: the leader has read everything it needs from the other CTAs
  if (rank != 0) return;

  const float m = sh.row_m, Z = sh.row_Z;
  if (sh.mode == kModeBad) {
    if (tid == 0) write_bad_row(p, row, rc.capture);
    return;
  }
  if (sh.mode == kModeFast) {
    if (finish_fast<DT, NT, BUF>(p, rc, cand, sh, sh.count, m, Z, sh.tau)) return;
  }
  __syncthreads();
  general_path<DT, NT, BUF>(p, rc, cand, sh, m, Z);
}

}  // namespace sfc
