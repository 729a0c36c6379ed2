// Fused sample · filter · capture kernel for one decode step (sm_103a).
//
// Grid: one CTA per row; or, for short batches, 2-8 CTAs per row, each streaming a slice: ordinary
// CTAs that publish their candidates and statistics in the caller's workspace, the last to arrive
// (an atomic ticket) merging them and finishing the row, or, with a small top-k bound, a
// thread-block cluster exchanging them through distributed shared memory. One HBM read of the
// logits per row element:
//   ring     thread 0 keeps a ring of NS shared-memory stages of SB bytes filled with bulk
//            asynchronous copies of the row (cp.async.bulk, completion on mbarriers; every wait is
//            bounded), so many bytes are in flight per CTA without holding them in registers.
//   sample   the first stages are evenly spaced chunks of the row; their 16-byte vector maxima are
//            histogrammed in bins of 1/8 logit below the sample maximum, and the bin where the
//            running count reaches ks gives tau, at most the ks-th largest sampled maximum. ks is a
//            high quantile of how many of the row's k largest logits the sample holds, so tau is a
//            lower bound of the row's k-th largest logit with overwhelming probability (exactly,
//            when the sample is the whole row), and the finish verifies it.
//   stream   each thread keeps online softmax statistics (running max, sum of 2^((x-m)c)) of the
//            vectors it reads from the stages, and one ballot per vector slot records in a bitmap
//            which vectors reach tau: no barrier, no atomic and no append in the loop.
//   gather   the marked vectors (read again, from L2) give the candidates, the logits >= tau, as
//            64-bit keys (key << 32 | ~id) in ascending id order.
//   finish   bf16 rows: exact value bins (code distances, or dense value ranks past 1024 codes),
//            one scan of counts and masses gives the top-k (ties kept), top-p and min-p cuts and
//            the renormaliser of S; a stable per-warp counting sort places S in canonical order;
//            Philox exponential race over S; packed output for capturing rows. f32 rows and the
//            bins' fallbacks: value buckets with in-bucket ranks, then a scan in canonical order; f32
//            rows that do not capture skip the sort (S as three tests on a candidate's key, the race
//            over the pool as it lies).
//   general  rows whose candidates do not fit on chip (top_k disabled or very large on a long
//            row, or a tie group larger than the buffer) are finished with a few more passes
//            over the row: a radix descent that finds the top-k / top-p threshold with integer
//            counts and fixed-point masses, a pass for |S|, its renormaliser and the race, and,
//            for capturing rows with a support larger than the buffer, two count-only descents
//            that pick the first W support members in canonical order.
//   modes    flags select greedy rows (T = 0: the lowest id among the largest logits, a width-1
//            support), positional top-k / top-p (S's last tie group cut to its lowest ids) and the
//            min-p-first order (top-p against the min-p survivors' mass); a row offset keys the
//            race on global row indices, so that a batch sharded over calls draws as one call.
//
// Method sources, by page title and section: prhub summary of SGLang PR #36630 (实现拆解 2-4,
// 关键源码片段: joint top-k / top-p thresholds, ties kept, keep-sets intersected, support = positive
// weights); "[Sampling] Stream sampling masks as per-request arrays" (Contract; Checks removed
// item 1: packed per-row arrays, OK/OVERFLOW); "vLLM Sampling Mask（Distribution Replay）深入解析"
// (工作原理 Step 1-2: temperature, min-p, top-k/top-p; finite survivors); "topk-subset-sampler"
// (The fix: one top-k candidate subset, exponential race).
#pragma once

#include <cstdint>

#include "sfc_device.cuh"

namespace sfc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFixedScale = 1099511627776.0f;  // 2^40: fixed-point scale of probability weights
constexpr int kSampleBins = 256;                 // sample histogram: bins of 1/kSampleScale logit
constexpr float kSampleScale = 8.f;
constexpr int kFinishBinsPerWarp = 256;          // bucket-sort bins of the finish, per warp of the CTA
constexpr int kMaxGroup = 512;                   // largest bin the in-bin rank counting takes
constexpr int kRowTimeout = -2;                  // row status: a bounded wait gave up
constexpr uint32_t kFlagGreedyT0 = 1u;           // SFC_FLAG_GREEDY_T0
constexpr uint32_t kFlagPositional = 2u;         // SFC_FLAG_POSITIONAL
constexpr uint32_t kFlagMinPFirst = 4u;          // SFC_FLAG_MIN_P_FIRST
constexpr uint32_t kFlagTestStall = 8u;          // SFC_FLAG_TEST_STALL
constexpr uint32_t kStallPolls = 8;              // the pass's wait limit under SFC_FLAG_TEST_STALL

enum : int { kModeFast = 0, kModeGeneral = 1, kModeBad = 2 };

struct Params {
  const void* logits;
  int64_t row_stride;  // elements
  int64_t V;
  int32_t B;
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
  uint32_t* support_mask;  // [B, ceil(V / 32)] or null: S as a bitmask, for capturing rows with |S| > W
  uint32_t flags;          // SFC_FLAG_* bits
  int32_t split;           // CTAs per row (a thread-block cluster): 1, 2, 4 or 8
  int64_t row_offset;      // added to a row's index in the race's counter (a batch sharded over calls)
  // A row split into `slices` ordinary CTAs (1: not split) that meet through the caller's workspace:
  uint32_t* tickets;       // [B] arrivals of a row's slices; zero between calls
  uint4* slice_rec;        // [B * slices] per slice: threshold key, maximum, sum, pool size
  uint64_t* slice_pool;    // [B * slices * slice_cap] per slice: its candidates (composite keys)
  int32_t slices;
  int32_t slice_cap;       // entries of one slice's pool
};


template <int NT>
struct Shared {
  BlockScratch<NT> sc;
  unsigned long long* mass;  // [256] in dynamic shared memory (the multi-pass finish only)
  int samp_d;       // sample-histogram bin of the ks-th largest sampled logit, or -1
  int n_ext;        // candidates among the unaligned head / ragged tail scalars
  uint64_t ext[16];
  int count;        // the multi-pass path's gather count
  int timed_out;    // a bounded wait gave up
  int pool_n;       // candidates reserved in the pool (the unordered gather)
  int issued;       // ring stages issued so far (the largest stage index + 1)
  int left[16];     // warps that have read the ring slot's current stage
  float row_m, row_Z;
  // finish results
  float zs;
  int bk, nk;
  // general path
  int n_sel;
  uint32_t d_prefix;
  int d_rem, d_ka, d_pa, d_done;
  unsigned long long d_mass_above, d_thr;
  int d_cnt_above;
  int gather_overflow;
  // a row split over a cluster, by slice rank (each slice stores its own entry into every CTA of
  // the cluster): threshold, statistics, pool size (-1: incomplete, -2: a wait gave up) and the
  // number of candidates it keeps
  uint32_t sx_tau[8];
  float sx_m[8], sx_Z[8];
  int sx_U[8], sx_cnt[8];
  int last;  // a slice of a split row: this CTA arrived last and finishes the row
};

// Per-row constants, identical in every thread of the CTA.
struct RowCtx {
  int row;
  uint32_t noise_row;  // the row's index in the race's counter: row_offset + row
  int64_t V;
  float T, invT, c, top_p, ln_min_p;
  int k;
  bool k_active, p_active, m_active, capture;
  bool greedy;      // temperature 0 under the greedy flag: the largest logit's lowest id, a width-1 support
  bool positional;  // top-k / top-p truncate the canonical order by position (ties may be cut)
  bool minp_first;  // min-p runs first: top-p's masses are renormalised over the min-p survivors M
  const unsigned char* rowp;
  int64_t head, nvec, body_end;  // the row: unaligned head scalars, 16-byte vectors, end of the vectors
  int64_t vec0, svec;            // this CTA's slice of the vectors: [vec0, vec0 + svec)
  int x_head, x_tail;            // head / tail scalars this CTA reads (the first / last slice)
};

// z - z_max = (x - m) / T, as a product with the row's reciprocal temperature (one division per row;
// within 1.5 ulp of the quotient, far inside the logprob tolerance and the min-p margin).
__device__ __forceinline__ float zrel_of(float x, float m, float invT) { return __fmul_rn(x - m, invT); }

// Race score of support member `id` at z - z_max = zr (one out-of-line copy: every finish calls it).
static __device__ __noinline__ float race_member_score(uint64_t seed, uint64_t step, uint32_t noise_row, uint32_t id,
                                                       float zr) {
  return race_score(zr, race_uniform(seed, step, noise_row, id));
}

// Outputs of a greedy row: the token, and for a capturing row the width-1 support {token} with
// log-probability 0 (one thread).
static __device__ __noinline__ void write_greedy_row(const Params& p, int row, bool capture, uint32_t token) {
  p.tokens[row] = static_cast<int32_t>(token);
  p.row_status[row] = 0;
  if (capture) {
    p.lengths[row] = 1;
    p.selected_logprob[row] = 0.f;
    p.support_ids[static_cast<int64_t>(row) * p.W] = static_cast<int32_t>(token);
    if (p.support_logprobs) p.support_logprobs[static_cast<int64_t>(row) * p.W] = 0.f;
  } else if (p.lengths) {
    p.lengths[row] = 0;
  }
}

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

// The exact support of an overflowing capturing row as a bitmask ("vLLM Sampling Mask（Distribution
// Replay）深入解析", 工作原理 Step 2: rows wider than the compact id buffer fall back to a packed
// bitmask): bit i % 32 of word i / 32 is set iff token i is in S. in_S(x, id) decides membership. On a 16-byte aligned row the threads read consecutive
// vectors (coalesced, U per thread in flight) and the lanes of a word merge their bits by shuffles;
// the rest of the row (unaligned rows, a ragged end) goes element by element.
template <int DT, int NT, typename F>
__device__ __noinline__ void write_support_mask(const Params& p, const RowCtx& rc, F&& in_S) {
  using E = Elem<DT>;
  constexpr int VEC = E::kVec;
  constexpr int VPW = 32 / VEC;  // vectors per mask word
  constexpr int U = 4;           // vectors in flight per thread
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t nwords = (rc.V + 31) / 32;
  uint32_t* out = p.support_mask + static_cast<int64_t>(rc.row) * nwords;
  int64_t nwf = 0;  // words built from whole aligned vectors
  if (rc.head == 0) {  // uniform
    const uint4* vb = reinterpret_cast<const uint4*>(rc.rowp);
    nwf = (rc.V / VEC) / VPW;
    const int64_t nvw = nwf * VPW;
    for (int64_t j0 = 0; j0 < nvw; j0 += static_cast<int64_t>(NT) * U) {  // uniform
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + u * NT + tid;
        v[u] = ld_stream(vb + min(j, nvw - 1));  // clamped: always a valid address
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + u * NT + tid;
        uint32_t b = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          b |= static_cast<uint32_t>(in_S(E::get(v[u], e), static_cast<uint32_t>((min(j, nvw - 1)) * VEC + e))) << e;
        b <<= VEC * (lane % VPW);  // vector j's place in word j / VPW (NT is a multiple of 32)
#pragma unroll
        for (int o = 1; o < VPW; o <<= 1) b |= __shfl_xor_sync(kFull, b, o);
        if (j < nvw && lane % VPW == 0) out[j / VPW] = b;
      }
    }
  }
  for (int64_t w = nwf + tid; w < nwords; w += NT) {  // the rest element by element
    const int64_t i0 = w * 32;
    uint32_t bits = 0;
    for (int b = 0; b < 32 && i0 + b < rc.V; ++b)
      bits |= static_cast<uint32_t>(in_S(E::load1(rc.rowp, i0 + b), static_cast<uint32_t>(i0 + b))) << b;
    out[w] = bits;
  }
}

// The same bitmask from S's members when they are all on chip (S[0..nS), composite keys): the row
// of the mask is cleared, then each member sets its bit (a global atomic OR).
template <int NT>
__device__ __noinline__ void write_support_mask_ids(const Params& p, const RowCtx& rc, const uint64_t* S, int nS) {
  const int64_t nwords = (rc.V + 31) / 32;
  uint32_t* out = p.support_mask + static_cast<int64_t>(rc.row) * nwords;
  for (int64_t w = threadIdx.x; w < nwords; w += NT) out[w] = 0;
  cta_sync<NT>();  // the cleared words come before any bit (one block, global memory)
  for (int i = threadIdx.x; i < nS; i += NT) {
    const uint32_t id = ckey_id(S[i]);
    atomicOr(&out[id >> 5], 1u << (id & 31));
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
// Streaming state of the row's CTA.
//
// The body is read in stages of SB bytes (chunk c = body vectors [c VS, (c+1) VS)). The first G
// stages are chunks from G evenly spaced stretches of the row: their vector maxima are the sample
// from which tau comes. The rest follow in order. No candidate is extracted while streaming:
// each warp marks, one ballot per vector slot, which of its vectors reach tau, in a bitmap with
// one bit per body vector; the finish reads the marked vectors again (from L2: the row has just
// streamed through it).
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int NS, int SB, int BITW, int GSN>
struct Streamer {
  using K = Keys<DT>;
  using E = Elem<DT>;
  static constexpr int VEC = E::kVec;
  static constexpr int VS = SB / 16;  // 16-byte vectors per stage
  static constexpr int UV = VS / NT;  // vectors per thread per stage
  static constexpr int NW = NT / 32;
  static constexpr int GS = GSN;  // sample stages at most
  static_assert(VS % NT == 0 && NS <= 16 && NW <= 32 && GSN >= 1 && GSN <= NS, "stage shapes");
  Shared<NT>& sh;
  unsigned char* ring;
  uint64_t* full;  // [NS] stage filled
  uint32_t* bits;  // [BITW] one bit per body vector: its maximum reaches tau
  float c;
  int k;
  bool k_active;
  int64_t V;
  const uint4* body;  // the row's 16-byte aligned body
  int64_t nvec;       // vectors in the body
  int nchunks;        // stages' worth of body
  int G, L;           // sample stages; the sample chunks are g L, g < G
  int depth;          // ring slots this row keeps in flight (1..NS)
  uint32_t head;      // token id of body element 0
  float m_t = -INFINITY, s_t = 0.f;  // online softmax state of this thread
  uint32_t tau = kKeyLowestFinite;   // candidate threshold (key) and its value
  float tau_f;
  float xe;  // one extra scalar (unaligned head / ragged tail), -inf if none
  uint32_t ide;
  bool has_xe;
  int n_extra;
  int64_t row_units;  // vectors and scalars of the whole row (this CTA may stream only a slice of it)
  bool bits_ok;  // the bitmap covers the body
  bool stalled;  // the test flag: stage 0 was never issued
  uint32_t polls = kWaitPolls;  // the pass's wait limit

  // The geometry of this CTA's part of the row: from the kernel's arguments alone, so that the first
  // stages can be issued before the row's parameters are loaded.
  __device__ Streamer(Shared<NT>& shr, unsigned char* rg, uint64_t* bars, uint32_t* bm, const RowCtx& r)
      : sh(shr), ring(rg), full(bars), bits(bm), depth(NS) {
    V = r.V;
    body = reinterpret_cast<const uint4*>(r.rowp + r.head * E::kBytes) + r.vec0;
    nvec = r.svec;
    nchunks = static_cast<int>((nvec + VS - 1) / VS);
    G = min(GS, nchunks);
    L = G > 0 ? nchunks / G : 1;
    head = static_cast<uint32_t>(r.head + r.vec0 * VEC);  // id of this slice's first vector element
    tau_f = K::value(tau);
    bits_ok = static_cast<int64_t>(nchunks) * (VS / 32) <= BITW;
    row_units = r.nvec + r.head + (r.V - r.body_end);
  }

  // The row's parameters, the ring depth it keeps in flight, the pass's wait limit and this thread's
  // extra scalar.
  __device__ void begin(const RowCtx& r, int dp, uint32_t wait_polls) {
    c = r.c;
    k = r.k;
    k_active = r.k_active;
    depth = dp;
    polls = wait_polls;
    const int tid = threadIdx.x;
    const int n_head = r.x_head, n_tail = r.x_tail;
    n_extra = n_head + n_tail;  // < 2 VEC <= NT
    has_xe = tid < n_extra;
    xe = -INFINITY;
    ide = 0;
    if (n_extra > 0) {  // uniform; the load is clamped to a valid index and masked by a select
      const int64_t idx = !has_xe ? (n_head > 0 ? 0 : r.body_end)
                                  : (tid < n_head ? tid : r.body_end + (tid - n_head));
      const float v = E::load1(r.rowp, idx);
      xe = has_xe ? v : -INFINITY;
      ide = static_cast<uint32_t>(idx);
    }
  }

  // Chunk read at stage s: the sample chunks first, then every other chunk in order.
  __device__ __forceinline__ int chunk_of(int s) const {
    if (s < G) return s * L;
    const int j = s - G;
    const int inner = G * (L - 1);  // non-sample chunks below G L
    return j < inner ? (j / (L - 1)) * L + j % (L - 1) + 1 : G * L + (j - inner);
  }

  // Start the bulk copy of stage s into ring slot `slot` (= s mod depth; one thread).
  __device__ __forceinline__ void issue(int s, int slot) {
    const int64_t v0 = static_cast<int64_t>(chunk_of(s)) * VS;
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(VS), nvec - v0)) * 16u;
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_load(ring + slot * SB, body + v0, bytes, &full[slot]);
  }
  // After a wait gave up (one thread): wait, with the full limit, for the copies still in flight, so
  // that none lands in shared memory after the CTA has exited. (A stalled stage 0 was never issued.)
  __device__ void drain() const {
    const int issued = sh.issued;
    for (int s = 0; s < depth && s < issued; ++s) {
      const int last = s + depth * ((issued - 1 - s) / depth);
      if (stalled && last == 0) continue;
      (void)mbar_wait(&full[s], static_cast<uint32_t>(last / depth) & 1u);
    }
  }

  // Read a stage (body chunk `chunk`, ring slot `slot`, that slot's use parity `ph`) into
  // registers (waiting for it unless `ready`). Returns the number of valid vectors, or -1 if the
  // wait gave up.
  // A wait that gives up does so for the whole warp (the warp's later ballots need every lane).
  __device__ __forceinline__ int read(int slot, uint32_t ph, int chunk, uint4 (&cur)[UV], bool ready) {
    const int tid = threadIdx.x;
    if (!ready && !__all_sync(kFull, mbar_wait(&full[slot], ph, polls))) {
      sh.timed_out = 1;
      return -1;
    }
    const int nv = static_cast<int>(min(static_cast<int64_t>(VS), nvec - static_cast<int64_t>(chunk) * VS));
    const uint4* st = reinterpret_cast<const uint4*>(ring + slot * SB);
    if (nv == VS) {  // uniform: only the body's last chunk is partial
#pragma unroll
      for (int u = 0; u < UV; ++u) cur[u] = st[u * NT + tid];
    } else {
#pragma unroll
      for (int u = 0; u < UV; ++u) {
        const int j = u * NT + tid;
        cur[u] = st[min(j, nv - 1)];  // clamped, unconditional
        if (!(j < nv)) cur[u] = E::neg_inf_vec();
      }
    }
    return nv;
  }

  // This warp is done with stage s (in ring slot `slot`); the last warp to leave refills the slot
  // with stage s + depth.
  __device__ __forceinline__ void release(int s, int slot) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      __threadfence_block();  // this warp's reads of the slot come before the refill
      if (atomicAdd(&sh.left[slot], 1) == NW - 1) {
        sh.left[slot] = 0;  // next used after full[slot] completes again, which the refill orders
        if (s + depth < nchunks) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          atomicMax(&sh.issued, s + depth + 1);
          issue(s + depth, slot);
        }
      }
    }
  }

  // Fold this thread's UV vectors of a stage into the statistics; vm[u] gets vector u's maximum.
  // NaN and +inf are not tested element by element: +inf becomes the maximum and NaN poisons the
  // sum, and the row is rejected from either.
  __device__ __forceinline__ void fold(const uint4 (&cur)[UV], float (&vm)[UV]) {
    float tmax = -INFINITY;
#pragma unroll
    for (int u = 0; u < UV; ++u) {
      vm[u] = E::vmax(cur[u]);
      tmax = fmaxf(tmax, vm[u]);
    }
    if (!(tmax <= m_t)) {
      const float mn = fmaxf(m_t, tmax);
      if (m_t > -INFINITY) s_t *= ex2_approx((m_t - mn) * c);
      m_t = mn;
    }
    const float nmc = m_t > -INFINITY ? -m_t * c : 0.f;  // 2^(x c - m c); while m = -inf every x is -inf
    if constexpr (DT == 0) {
      // bf16: the two elements of each 32-bit word widen into the two lanes of a packed f32x2 FMA;
      // per vector the eight weights meet in a fixed tree of packed adds, into two running sums.
      const uint64_t c2 = pack_f2(c, c), n2 = pack_f2(nmc, nmc);
      uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
      for (int u = 0; u < UV; ++u) {
        const uint32_t wd[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
        uint64_t q[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint64_t x2 = pack_f2(__uint_as_float(wd[w] << 16), __uint_as_float(wd[w] & 0xFFFF0000u));
          float a0, a1;
          unpack_f2(ffma_f2(x2, c2, n2), a0, a1);
          q[w] = pack_f2(ex2_approx(a0), ex2_approx(a1));
        }
        acc2[u & 1] = fadd_f2(acc2[u & 1], fadd_f2(fadd_f2(q[0], q[2]), fadd_f2(q[1], q[3])));
      }
      float s0, s1, s2, s3;
      unpack_f2(acc2[0], s0, s1);
      unpack_f2(acc2[1], s2, s3);
      s_t += (s0 + s1) + (s2 + s3);
    } else {
      float acc[2] = {0.f, 0.f};
#pragma unroll
      for (int u = 0; u < UV; ++u) {  // a short tree per vector, two running sums
        float t[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) t[e] = ex2_approx(fmaf(E::get(cur[u], e), c, nmc));
#pragma unroll
        for (int h = VEC / 2; h > 0; h >>= 1) {
#pragma unroll
          for (int e = 0; e < h; ++e) t[e] += t[e + h];
        }
        acc[u & 1] += t[0];
      }
      s_t += acc[0] + acc[1];
    }
  }

  // Bitmap words of a chunk: one ballot per vector slot (bit i of a word: the warp's lane i).
  __device__ __forceinline__ void mark(int chunk, const float (&vm)[UV]) {
    const int tid = threadIdx.x;
    const int base = chunk * VS + (tid & ~31);
#pragma unroll
    for (int u = 0; u < UV; ++u) {
      const unsigned b = __ballot_sync(kFull, vm[u] >= tau_f);  // invalid lanes are -inf
      if ((tid & 31) == 0 && bits_ok) bits[(base + u * NT) >> 5] = b;
    }
  }

  // The extra scalar of this thread (if any): statistics only; it is a candidate if >= tau.
  __device__ __forceinline__ void fold_extra() {
    if (!(xe <= m_t)) {
      const float mn = fmaxf(m_t, xe);
      if (m_t > -INFINITY) s_t *= ex2_approx((m_t - mn) * c);
      m_t = mn;
    }
    s_t += ex2_approx(fmaf(xe, c, m_t > -INFINITY ? -m_t * c : 0.f));  // -inf gives 0
  }

  // tau from the sample (the vector maxima of the first G stages and the extra scalars), in bins
  // of 1/8 logit below floor(8 max): the bin where the running count from the top reaches ks has
  // lower edge tv <= the ks-th largest sampled maximum. The row's k-1 largest logits lie in at
  // most k-1 vectors (or scalars); with f the sampled fraction of the ROW's vectors, about
  // Poisson(lam) of them are sampled, lam = (k-1) f. If tv exceeded the row's k-th largest logit,
  // at least ks of those vectors would be sampled; ks = lam + 5.3 sqrt(lam) + 6 makes that rarer
  // than about 1e-7. When the sample is the whole row, ks = k: k vectors reach tv, so k logits do.
  // A CTA that streams one slice of a row samples at most that slice, so its ks is about k / slices
  // and its threshold is a lower bound of the row's (not the slice's) k-th largest logit: the
  // largest of the slices' thresholds is then checked against the merged candidates.
  __device__ void threshold(const float (&keep)[GS][UV], int n_sampled) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    float mx = xe;
#pragma unroll
    for (int g = 0; g < GS; ++g) {
#pragma unroll
      for (int u = 0; u < UV; ++u) mx = fmaxf(mx, keep[g][u]);  // unsampled slots are -inf
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    for (int i = tid; i < 256; i += NT) sh.sc.hist[i] = 0;
    if (lane == 0) sh.sc.red_f[w] = mx;
    cta_sync<NT>();
    float m0 = sh.sc.red_f[0];
    for (int i = 1; i < NW; ++i) m0 = fmaxf(m0, sh.sc.red_f[i]);
    const bool usable = m0 > -1048576.f && m0 < 1048576.f;  // finite, and small enough for integer bins
    const int top = usable ? static_cast<int>(floorf(m0 * kSampleScale)) : 0;
    if (usable) {
      const float lo_bin = static_cast<float>(top - kSampleBins);
      auto add = [&](float x) {
        const float fx = floorf(x * kSampleScale);  // NaN and -inf fail the test below
        if (fx > lo_bin && fx <= static_cast<float>(top)) atomicAdd(&sh.sc.hist[top - static_cast<int>(fx)], 1u);
      };
      add(xe);
#pragma unroll
      for (int g = 0; g < GS; ++g) {
#pragma unroll
        for (int u = 0; u < UV; ++u) add(keep[g][u]);
      }
    }
    cta_sync<NT>();
    const int64_t units = row_units;
    const int64_t sampled = static_cast<int64_t>(n_sampled) + n_extra;
    int ks;
    if (sampled >= units) {
      ks = k;
    } else {
      const float lam = static_cast<float>(k) * static_cast<float>(sampled) / static_cast<float>(units);
      ks = static_cast<int>(ceilf(lam + 5.3f * sqrtf(lam) + 6.f));
    }
    const int cnt = tid < kSampleBins ? static_cast<int>(sh.sc.hist[tid]) : 0;
    int total;
    const int ex = Block<NT>::excl_scan_int(cnt, sh.sc.red_i, total);
    if (usable && cnt > 0 && ex < ks && ex + cnt >= ks) sh.samp_d = tid;
    cta_sync<NT>();
    const int d = sh.samp_d;
    if (d >= 0) {
      const float tv = static_cast<float>(top - d) / kSampleScale;  // exact: |top - d| < 2^24
      uint32_t t = K::key(tv);
      if (K::value(t) > tv) t -= (DT == 0 ? 0x10000u : 1u);  // bf16 keys round negative values up
      tau = max(t, kKeyLowestFinite);
      tau_f = K::value(tau);
    }
  }

  // The pass over the row. Returns false if a bounded wait gave up.
  __device__ bool stream() {
    float keep[GS][UV];
    int n_sampled = 0;  // valid vectors among the sample stages
    int slot = 0;       // stage s's ring slot: s mod depth, and that slot's use parity
    uint32_t ph = 0;
    auto next_slot = [&]() {
      if (++slot == depth) {
        slot = 0;
        ph ^= 1u;
      }
    };
    bool failed = false;  // a wait of this warp gave up: it reads no further stage
#pragma unroll
    for (int g = 0; g < GS; ++g) {
#pragma unroll
      for (int u = 0; u < UV; ++u) keep[g][u] = -INFINITY;
      if (g < G && !failed) {  // warp-uniform
        uint4 cur[UV];
        const int nv = read(slot, ph, g * L, cur, false);
        if (nv < 0) {
          failed = true;
        } else {
          release(g, slot);
          next_slot();
          n_sampled += nv;
          fold(cur, keep[g]);
        }
      }
    }
    // The threshold's barriers need every thread: the block decides together whether the pass goes on.
    if (cta_sync_or<NT>(failed)) return false;
    if (k_active) threshold(keep, n_sampled);
    if (xe >= tau_f) sh.ext[atomicAdd(&sh.n_ext, 1)] = make_ckey(K::key(xe), ide);  // at most 2 VEC - 2
#pragma unroll
    for (int g = 0; g < GS; ++g) {
      if (g < G) mark(g * L, keep[g]);
    }
    // The other chunks in order, skipping the sample chunks g L (g < G); r tracks c mod L.
    int c = L > 1 ? 1 : G, r = L > 1 ? 1 : 0;
    for (int s = G; s < nchunks; ++s) {
      uint4 cur[UV];
      float vm[UV];
      if (read(slot, ph, c, cur, false) < 0) return false;
      release(s, slot);
      next_slot();
      fold(cur, vm);
      mark(c, vm);
      ++c;
      if (++r == L) r = 0;
      if (r == 0 && c < G * L) {
        ++c;
        r = L > 1 ? 1 : 0;
      }
    }
    return true;
  }
};

// ------------------------------------------------------------------------------------------
// From K in canonical order (cand[0..n), the top-k tie groups): top-p and min-p cuts, the
// renormaliser of S, the exponential race over S and the outputs.
// ------------------------------------------------------------------------------------------
template <int DT, int NT>
__device__ __noinline__ void finish_sorted(const Params& p, const RowCtx rc, const uint64_t* cand, Shared<NT>& sh,
                                           int n, float m, float Z) {
  using K = Keys<DT>;
  const int tid = threadIdx.x;
  if (rc.positional && rc.k_active) n = min(n, rc.k);  // K: the first k positions
  // Exclusive scan of the weights 2^((x-m)c) in canonical order; cut at the first tie group
  // whose mass above exceeds top_p * Z (positionally: the first position whose own mass before
  // does), or whose z - z_max falls below ln(min_p). Warp w owns the
  // run [w CW, (w + 1) CW) and its lanes take consecutive entries (no bank conflicts); a shuffle
  // scan per round of 32 carries the prefix.
  constexpr int NW = NT / 32;
  const int lane = tid & 31, wp = tid >> 5;
  const int C = (n + NT - 1) / NT;
  const int CW = 32 * C;
  const int r0 = min(wp * CW, n), r1 = min(r0 + CW, n);
  auto weight = [&](int i) { return ex2_approx((K::value(ckey_key(cand[i])) - m) * rc.c); };
  float part = 0.f;
  for (int i = r0 + lane; i < r1; i += 32) part += weight(i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFull, part, o);
  if (lane == 0) sh.sc.red_f[wp] = part;
  cta_sync<NT>();
  float off = 0.f, total = 0.f;
  for (int v = 0; v < NW; ++v) {
    const float t = sh.sc.red_f[v];
    off += v < wp ? t : 0.f;
    total += t;
  }
  const float thr = rc.top_p * Z;
  // The warp's scan: calls f(i, mass before i) for each of its entries in order.
  auto walk = [&](int end, auto&& f) {
    float base = off;
    for (int j0 = r0; j0 < end; j0 += 32) {  // warp-uniform
      const int i = j0 + lane;
      const float wi = i < end ? weight(i) : 0.f;
      const float incl = warp_incl_scan_f(wi);
      if (i < end) f(i, base + incl - wi);
      base += __shfl_sync(kFull, incl, 31);
    }
  };
  int cut = n;
  walk(r1, [&](int i, float pre) {
    const uint32_t key = ckey_key(cand[i]);
    const bool gstart = (i == 0) || ckey_key(cand[i - 1]) != key;
    if ((gstart || rc.positional) && cut == n) {
      if (rc.p_active && pre > thr) cut = i;
      if (rc.m_active && zrel_of(K::value(key), m, rc.invT) < rc.ln_min_p) cut = i;
    }
  });
  cut = Block<NT>::min_int(cut, sh.sc.red_i);
  const int nS = cut;  // >= 1: the first group always passes
  if (nS == n) {
    if (tid == 0) sh.zs = total;
  } else if (wp == nS / CW) {  // the warp holding entry nS: its mass before nS
    walk(min(r1, nS + 1), [&](int i, float pre) {
      if (i == nS) sh.zs = pre;
    });
  }
  cta_sync<NT>();
  const float logZS = logf(sh.zs);
  if (rc.greedy) {  // cand[0]: the lowest id of the largest value
    if (tid == 0) write_greedy_row(p, rc.row, rc.capture, ckey_id(cand[0]));
    return;
  }

  // Exponential race over S.
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
  if constexpr (DT == 1) {
    // float rows (wide supports: many members per thread): four members at a time, so that four
    // independent Philox chains overlap
    constexpr int RU = 4;
    for (int i0 = tid; i0 < nS; i0 += NT * RU) {
      float sc[RU], xs[RU];
      uint32_t idv[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const uint64_t ck = cand[min(i0 + u * NT, nS - 1)];
        xs[u] = K::value(ckey_key(ck));
        idv[u] = ckey_id(ck);
        sc[u] = race_score(zrel_of(xs[u], m, rc.invT), race_uniform(p.seed, p.step, rc.noise_row, idv[u]));
      }
#pragma unroll
      for (int u = 0; u < RU; ++u)
        if (i0 + u * NT < nS && race_better(sc[u], idv[u], best, bid)) { best = sc[u]; bid = idv[u]; bx = xs[u]; }
    }
  } else {
    for (int i = tid; i < nS; i += NT) {
      const uint64_t ck = cand[i];
      const float x = K::value(ckey_key(ck));
      const uint32_t id = ckey_id(ck);
      const float sc = race_member_score(p.seed, p.step, rc.noise_row, id, zrel_of(x, m, rc.invT));
      if (race_better(sc, id, best, bid)) { best = sc; bid = id; bx = x; }
    }
  }
  Block<NT>::race_argmax(best, bid, bx, sh.sc.red_f, sh.sc.red_u, sh.sc.red_x);

  if (tid == 0) {
    p.tokens[rc.row] = static_cast<int32_t>(bid);
    if (rc.capture) {
      p.lengths[rc.row] = nS;
      p.row_status[rc.row] = nS > p.W ? 1 : 0;
      p.selected_logprob[rc.row] = zrel_of(bx, m, rc.invT) - logZS;
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
      if (lps) lps[i] = zrel_of(K::value(ckey_key(ck)), m, rc.invT) - logZS;
    }
    if (p.support_mask && nS > p.W) write_support_mask_ids<NT>(p, rc, cand, nS);  // uniform
  }
}

// ------------------------------------------------------------------------------------------
// Finish from a list of candidates on chip, sorted by radix select, compaction and merge sort:
// cand[0..n) holds every row token >= tau_floor (every finite token when top-k is off).
// Returns false (nothing written) if tau_floor overshot the k-th largest or K does not fit.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int BUF>
__device__ __noinline__ bool finish_fast(const Params& p, const RowCtx rc, uint64_t* cand, Shared<NT>& sh, int n,
                                         float m, float Z, uint32_t tau_floor) {
  using K = Keys<DT>;
  constexpr int SORT_E = (NT >= 512) ? 16 : 8;  // register-sorted run length of the merge sort
  constexpr int SORT_CAP = (BUF & (BUF - 1)) == 0 ? BUF : (1 << (31 - __builtin_clz(BUF)));
  // If the buffer's k-th largest is >= tau_floor, the top-k with ties is complete; otherwise the
  // threshold estimate was too high and the multi-pass path takes the row.
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
  finish_sorted<DT, NT>(p, rc, cand, sh, n, m, Z);
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
    for (int i = threadIdx.x; i < kWarps * 256; i += NT) sh.sc.whist[i] = 0;
    cta_sync<NT>();
    row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
      bool ok = valid && sel(x, id);
      const uint32_t v = val(x, id);
      if (pass > 0) ok = ok && (v >> (shift + 8)) == (prefix >> (shift + 8));
      warp_hist_inc(sh.sc.whist + warp * 256, (v >> shift) & 0xFFu, ok);
    });
    cta_sync<NT>();
    for (int b = threadIdx.x; b < 256; b += NT) {
      uint32_t t = 0;
      for (int w = 0; w < kWarps; ++w) t += sh.sc.whist[w * 256 + b];
      sh.sc.hist[b] = t;
    }
    cta_sync<NT>();
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
    cta_sync<NT>();
    prefix = sh.d_prefix;
    rem = sh.d_rem;
    above = sh.d_cnt_above;
    cta_sync<NT>();
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
  cta_sync<NT>();
  for (int level = 0; level < K::kDigitPasses; ++level) {
    if (sh.d_done) break;
    const int shift = 24 - 8 * level;
    const uint32_t prefix = sh.d_prefix;
    const bool pa = sh.d_pa;
    // Warp-private count and fixed-point mass histograms (the mass ones live in the candidate
    // buffer, unused until the gather); integer sums, so the order of the adds does not matter.
    unsigned long long* wmass = reinterpret_cast<unsigned long long*>(cand);
    for (int i = tid; i < kWarps * 256; i += NT) {
      sh.sc.whist[i] = 0;
      wmass[i] = 0;
    }
    cta_sync<NT>();
    row_pass<DT, NT>(rc, [&](float x, uint32_t, bool valid) {
      const uint32_t key = K::key(x);
      // min-p-first: the tokens min-p drops are out of both counts and masses (they were -inf)
      bool ok = valid && x > -INFINITY && (!rc.minp_first || zrel_of(x, m, rc.invT) >= rc.ln_min_p);
      if (level > 0) ok = ok && (key >> (shift + 8)) == (prefix >> (shift + 8));
      const uint32_t d = (key >> shift) & 0xFFu;
      warp_hist_inc(sh.sc.whist + warp * 256, d, ok);
      if (pa && ok) atomicAdd(&wmass[warp * 256 + d], static_cast<unsigned long long>(__float2ull_rn(ex2_approx((x - m) * c) * kFixedScale)));
    });
    cta_sync<NT>();
    for (int b = tid; b < 256; b += NT) {
      uint32_t t = 0;
      unsigned long long mm = 0;
      for (int w = 0; w < kWarps; ++w) {
        t += sh.sc.whist[w * 256 + b];
        mm += wmass[w * 256 + b];
      }
      sh.sc.hist[b] = t;
      sh.mass[b] = mm;
    }
    cta_sync<NT>();
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
    cta_sync<NT>();
  }
  // With neither constraint ever active the threshold stays 0: every finite token passes.
  const uint32_t tau = sh.d_prefix;
  cta_sync<NT>();

  auto in_S = [&](float x) -> bool {
    if (!(x > -INFINITY)) return false;
    if (K::key(x) < tau) return false;
    if (rc.m_active && zrel_of(x, m, rc.invT) < rc.ln_min_p) return false;
    return true;
  };

  if (rc.greedy) {  // the lowest id among the largest logits
    uint32_t low = 0xFFFFFFFFu;
    row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
      if (valid && x == m && id < low) low = id;
    });
    const int lowest = Block<NT>::min_int(static_cast<int>(min(low, 0x7FFFFFFFu)), sh.sc.red_i);  // ids < 2^31
    if (tid == 0) write_greedy_row(p, rc.row, rc.capture, static_cast<uint32_t>(lowest));
    return;
  }

  // Positional top-k / top-p cut only the last tie group of the joint S, to its lowest ids: count
  // that group and the mass above it, keep its first j members and find the j-th lowest id.
  uint32_t key_last = 0, idinv_last = 0;  // with idinv_last = 0 every member of the group stays
  if (rc.positional && (rc.k_active || rc.p_active)) {
    int n_loc = 0;
    int kmin = 0x7FFFFFFF;
    row_pass<DT, NT>(rc, [&](float x, uint32_t, bool valid) {
      if (valid && in_S(x)) {
        ++n_loc;
        kmin = min(kmin, static_cast<int>(K::key(x) ^ 0x80000000u));
      }
    });
    const int n_joint = Block<NT>::sum_int(n_loc, sh.sc.red_i);
    key_last = static_cast<uint32_t>(Block<NT>::min_int(kmin, sh.sc.red_i)) ^ 0x80000000u;
    int g_loc = 0;
    float above = 0.f;
    row_pass<DT, NT>(rc, [&](float x, uint32_t, bool valid) {
      if (!(valid && in_S(x))) return;
      if (K::key(x) == key_last) ++g_loc;
      else above += ex2_approx((x - m) * c);
    });
    const int g_last = Block<NT>::sum_int(g_loc, sh.sc.red_i);
    const float mass_above = Block<NT>::sum(above, sh.sc.red_f);
    int keep = g_last;
    if (rc.k_active) keep = min(keep, rc.k - (n_joint - g_last));
    if (rc.p_active) {  // member j's own mass before: mass_above + j w
      float ZP = Z;
      if (rc.minp_first) {  // M's mass
        float zm = 0.f;
        row_pass<DT, NT>(rc, [&](float x, uint32_t, bool valid) {
          if (valid && x > -INFINITY && zrel_of(x, m, rc.invT) >= rc.ln_min_p) zm += ex2_approx((x - m) * c);
        });
        ZP = Block<NT>::sum(zm, sh.sc.red_f);
      }
      const float w = ex2_approx((K::value(key_last) - m) * c);
      const float q = (rc.top_p * ZP - mass_above) / w;
      keep = min(keep, q < 0.f ? 0 : (q >= static_cast<float>(g_last) ? g_last : static_cast<int>(floorf(q)) + 1));
    }
    keep = max(keep, 1);
    if (keep < g_last) {
      int dummy = 0;
      idinv_last = general_descent_count<DT, NT>(
          rc, sh, keep, 4, [&](float x, uint32_t) { return in_S(x) && K::key(x) == key_last; },
          [&](float, uint32_t id) { return ~id; }, dummy);
    }
  }
  auto in_S2 = [&](float x, uint32_t id) -> bool {
    return in_S(x) && (idinv_last == 0 || K::key(x) != key_last || ~id >= idinv_last);
  };

  // 2. |S|, its renormaliser, the race; gather S when the row captures and S fits.
  if (tid == 0) {
    sh.count = 0;
    sh.gather_overflow = 0;
  }
  cta_sync<NT>();
  int n_loc = 0;
  float zs = 0.f, zc = 0.f;
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
  row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
    const bool ok = valid && in_S2(x, id);
    if (rc.capture) warp_append(cand, &sh.count, SORT_CAP, make_ckey(K::key(x), id), ok);  // collective first
    if (!ok) return;
    ++n_loc;
    const float y = ex2_approx((x - m) * c) - zc;
    const float t = zs + y;
    zc = (t - zs) - y;
    zs = t;
    const float sc = race_member_score(p.seed, p.step, rc.noise_row, id, zrel_of(x, m, rc.invT));
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
      p.selected_logprob[rc.row] = zrel_of(bx, m, rc.invT) - logZS;
    } else {
      p.row_status[rc.row] = 0;
      if (p.lengths) p.lengths[rc.row] = 0;
    }
  }
  if (!rc.capture) return;
  if (p.support_mask && nS > p.W) write_support_mask<DT, NT>(p, rc, in_S2);  // uniform
  cta_sync<NT>();

  // 3. The first min(|S|, W) members in canonical order.
  const int n_out = min(nS, p.W);
  if (nS > SORT_CAP) {
    // W-th largest key within S, then the lowest ids among the tokens tied at it.
    int c_gt = 0;
    const uint32_t tW = general_descent_count<DT, NT>(
        rc, sh, n_out, K::kDigitPasses, [&](float x, uint32_t id) { return in_S2(x, id); },
        [&](float x, uint32_t) { return K::key(x); }, c_gt);
    int dummy = 0;
    const uint32_t idinvW = general_descent_count<DT, NT>(
        rc, sh, n_out - c_gt, 4, [&](float x, uint32_t id) { return in_S2(x, id) && K::key(x) == tW; },
        [&](float, uint32_t id) { return ~id; }, dummy);
    if (tid == 0) sh.count = 0;
    cta_sync<NT>();
    row_pass<DT, NT>(rc, [&](float x, uint32_t id, bool valid) {
      const uint32_t key = K::key(x);
      const bool ok = valid && in_S2(x, id) && (key > tW || (key == tW && ~id >= idinvW));
      warp_append(cand, &sh.count, SORT_CAP, make_ckey(key, id), ok);
    });
    cta_sync<NT>();
  }
  const int n_have = min(sh.count, SORT_CAP);
  cta_sync<NT>();
  cand = block_sort_desc<NT, SORT_E>(cand, n_have, BUF);
  int32_t* ids = p.support_ids + static_cast<int64_t>(rc.row) * p.W;
  float* lps = p.support_logprobs ? p.support_logprobs + static_cast<int64_t>(rc.row) * p.W : nullptr;
  for (int i = tid; i < n_out; i += NT) {
    const uint64_t ck = cand[i];
    ids[i] = static_cast<int32_t>(ckey_id(ck));
    if (lps) lps[i] = zrel_of(K::value(ckey_key(ck)), m, rc.invT) - logZS;
  }
}

// ------------------------------------------------------------------------------------------
// The bucket finish of a row that does not capture (and is neither greedy, positional nor in the
// min-p-first order): it needs only the token, so S is found as three tests on a candidate's key,
// each the set of tie groups before a cut in canonical order, and the race runs over the pool as it
// lies. K: key >= the k-th largest key (its tie group kept), the k-th largest found by ranking bin bk
// alone. P: the first tie group whose mass of larger logits exceeds top_p Z and every group after it
// leave; the bins' fixed-point masses (integer sums: the same in any order) locate the bin c where
// the cumulative mass first exceeds top_p Z, and only bin c's members are compared with one another.
// M: z - z_max >= ln(min_p). The bins (b(x), cnt[], fil[]: counts and exclusive starts, bins up to
// bk holding kk's tie group) are those of finish_bucket; scratch: the pool area behind pool[0..U),
// bk + 1 + 2 kMaxGroup + NT / 32 entries.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int NB>
__device__ __noinline__ void finish_unsorted(const Params& p, const RowCtx rc, const uint64_t* cand, Shared<NT>& sh,
                                             int U, float m, float Z, float inv, int kk, int bk) {
  using K = Keys<DT>;
  constexpr int PB = NB / NT;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint16_t* cnt = reinterpret_cast<const uint16_t*>(sh.sc.whist);
  const uint16_t* fil = cnt + NB;
  // scratch behind the pool: bin masses [bk + 1], bin bk's members, bin c's members, warp sums
  uint64_t* bm = const_cast<uint64_t*>(cand) + U;
  uint64_t* mk = bm + bk + 1;
  uint64_t* mc = mk + kMaxGroup;
  uint64_t* wsum = mc + kMaxGroup;
  auto bin_of = [&](uint64_t e) -> int {
    const float x = K::value(ckey_key(e));
    return min(static_cast<int>((m - x) * inv), NB - 1);
  };
  auto fixed_weight = [&](uint64_t e) -> uint64_t {  // 2^((x - m)c) <= 1 in units of 2^-40
    return static_cast<uint64_t>(__float2ull_rn(ex2_approx((K::value(ckey_key(e)) - m) * rc.c) * kFixedScale));
  };
  const bool pa = rc.p_active;
  if (tid == 0) {
    sh.count = 0;
    sh.n_sel = 0;
    sh.d_prefix = 0u;  // the k-th largest key
    sh.d_thr = 0ull;   // P's largest excluded key in bin c
  }
  if (pa)
    for (int i = tid; i <= bk; i += NT) bm[i] = 0ull;
  cta_sync<NT>();
  // bin bk's members; the masses of bins up to bk
  for (int i = tid; i < U; i += NT) {
    const uint64_t e = cand[i];
    const int b = bin_of(e);
    if (b == bk) mk[atomicAdd(&sh.count, 1)] = e;  // cnt[bk] <= kMaxGroup of them
    if (pa && b <= bk) atomicAdd(reinterpret_cast<unsigned long long*>(&bm[b]), static_cast<unsigned long long>(fixed_weight(e)));
  }
  cta_sync<NT>();
  // the k-th largest key: the member of bin bk with kk - 1 - fil[bk] larger members (composite keys
  // are distinct, so exactly one member has that rank)
  const int gk = cnt[bk], want = kk - 1 - static_cast<int>(fil[bk]);
  for (int i = tid; i < gk; i += NT) {
    const uint64_t e = mk[i];
    int r = 0;
    for (int j = 0; j < gk; ++j) r += mk[j] > e ? 1 : 0;
    if (r == want) sh.d_prefix = ckey_key(e);
  }
  // P's cut bin: the first bin whose cumulative mass exceeds top_p Z (thread t owns bins t PB ..)
  int c = NB;
  const double thr = static_cast<double>(rc.top_p) * static_cast<double>(Z) * static_cast<double>(kFixedScale);
  if (pa) {  // uniform
    uint64_t run = 0;
#pragma unroll
    for (int j = 0; j < PB; ++j) {
      const int b = tid * PB + j;
      if (b <= bk) run += bm[b];
    }
    uint64_t inc = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) wsum[w] = inc;
    cta_sync<NT>();
    uint64_t cum = inc - run;
    for (int v = 0; v < w; ++v) cum += wsum[v];
    int mine = NB;
    uint64_t before_mine = 0;
#pragma unroll
    for (int j = 0; j < PB; ++j) {
      const int b = tid * PB + j;
      if (b <= bk && mine == NB) {
        if (static_cast<double>(cum + bm[b]) > thr) {
          mine = b;
          before_mine = cum;
        }
        cum += bm[b];
      }
    }
    c = Block<NT>::min_int(mine, sh.sc.red_i);
    if (c < NB && mine == c) sh.d_mass_above = before_mine;  // the thread that owns bin c
  }
  cta_sync<NT>();
  const uint32_t key_k = sh.d_prefix;
  uint32_t key_p = 0u;  // in bin c, the keys of P are those > key_p (0: all of bin c)
  if (c < NB) {  // uniform: bin c's members, and the largest key whose larger logits' mass exceeds top_p Z
    const uint64_t before = sh.d_mass_above;
    for (int i = tid; i < U; i += NT) {
      const uint64_t e = cand[i];
      if (bin_of(e) == c) mc[atomicAdd(&sh.n_sel, 1)] = e;  // cnt[c] <= kMaxGroup of them
    }
    cta_sync<NT>();
    const int gc = cnt[c];
    for (int i = tid; i < gc; i += NT) {
      const uint32_t ke = ckey_key(mc[i]);
      uint64_t mb = before;
      for (int j = 0; j < gc; ++j)
        if (ckey_key(mc[j]) > ke) mb += fixed_weight(mc[j]);
      if (static_cast<double>(mb) > thr) atomicMax(reinterpret_cast<unsigned long long*>(&sh.d_thr), static_cast<unsigned long long>(ke));
    }
    cta_sync<NT>();
    key_p = static_cast<uint32_t>(sh.d_thr);
  }
  // the race over S = K, P and M, the pool as it lies
  auto in_s = [&](uint64_t e, float zr) {
    const uint32_t key = ckey_key(e);
    const int b = bin_of(e);
    return key >= key_k && (b < c || (b == c && key > key_p)) && (!rc.m_active || zr >= rc.ln_min_p);
  };
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
  if constexpr (DT == 1) {  // float rows: four entries at a time, four independent Philox chains
    constexpr int RU = 4;
    for (int i0 = tid; i0 < U; i0 += NT * RU) {
      float sc[RU], xs[RU];
      uint32_t idv[RU];
      bool ok[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int i = i0 + u * NT;
        const uint64_t e = cand[min(i, U - 1)];
        xs[u] = K::value(ckey_key(e));
        idv[u] = ckey_id(e);
        const float zr = zrel_of(xs[u], m, rc.invT);
        ok[u] = i < U && in_s(e, zr);
        sc[u] = race_score(zr, race_uniform(p.seed, p.step, rc.noise_row, idv[u]));
      }
#pragma unroll
      for (int u = 0; u < RU; ++u)
        if (ok[u] && race_better(sc[u], idv[u], best, bid)) {
          best = sc[u];
          bid = idv[u];
          bx = xs[u];
        }
    }
  } else {
    for (int i = tid; i < U; i += NT) {
      const uint64_t e = cand[i];
      const float x = K::value(ckey_key(e));
      const float zr = zrel_of(x, m, rc.invT);
      if (in_s(e, zr)) {
        const uint32_t id = ckey_id(e);
        const float sc = race_member_score(p.seed, p.step, rc.noise_row, id, zr);
        if (race_better(sc, id, best, bid)) {
          best = sc;
          bid = id;
          bx = x;
        }
      }
    }
  }
  Block<NT>::race_argmax(best, bid, bx, sh.sc.red_f, sh.sc.red_u, sh.sc.red_x);
  if (tid == 0) {
    p.tokens[rc.row] = static_cast<int32_t>(bid);
    p.row_status[rc.row] = 0;
    if (p.lengths) p.lengths[rc.row] = 0;
  }
}

// ------------------------------------------------------------------------------------------
// Finish from the row's candidates gathered in pool[0..U) (every row token >= tau, or every
// finite token when tau is the lowest key), by a bucket sort that stops at the k-th largest.
// The pool area holds CAP entries.
//
// Bins are a monotone function of the logit: b(x) = min(floor((m - x) * (NB-1) / (m - lo)), NB-1)
// with m the row maximum and lo at most the pool minimum (the minimum, or tau's value), so larger
// logits never land in later bins and equal logits share a bin. Bin counts and their exclusive scan
// locate the bin holding the k-th largest; only the bins up to it are placed, and inside a bin an
// entry's position is the number of members with a larger composite key (logit key, then lower id).
// The tie group of the k-th largest then closes K. A float row that does not capture stops after the
// bin counts and takes finish_unsorted instead.
// Returns 1 when the row is finished, 0 when this path cannot take it (pool[0..U) untouched) and
// -1 when tau overshot the row's k-th largest (the multi-pass path must take the row).
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int CAP>
__device__ __noinline__ int finish_bucket(const Params& p, const RowCtx rc, uint64_t* cand, Shared<NT>& sh, int U,
                                          float m, float Z, float lo, uint32_t tau) {
  using K = Keys<DT>;
  constexpr int NB = (NT / 32) * kFinishBinsPerWarp;  // the counters fill the warp histograms
  constexpr int PB = NB / NT;  // consecutive bins per thread in the scan
  // 16-bit counters (bins hold at most CAP < 65536 entries), two to a word: counts, then fill positions
  static_assert(NB % NT == 0 && (NT / 32) * 256 * 2 >= 2 * NB && CAP < 65536, "the bin counters live in the warp histograms");
  const int tid = threadIdx.x;
  uint16_t* cnt = reinterpret_cast<uint16_t*>(sh.sc.whist);
  uint16_t* fil = cnt + NB;
  uint32_t* cnt32 = sh.sc.whist;
  uint32_t* fil32 = cnt32 + NB / 2;
  int kk;
  if (rc.k_active && rc.k <= U) {
    kk = rc.k;
  } else if (rc.k_active && tau > kKeyLowestFinite) {
    return -1;  // fewer than k tokens >= tau
  } else {
    kk = U;  // every finite token is in the pool: K is all of them
  }
  const float range = m - lo;
  const float inv = (range > 0.f && range < INFINITY) ? static_cast<float>(NB - 1) / range : 0.f;
  auto bin_of = [&](uint64_t e) -> int {
    const float x = K::value(ckey_key(e));
    return min(static_cast<int>((m - x) * inv), NB - 1);
  };
  for (int i = tid; i < NB / 2; i += NT) cnt32[i] = 0u;
  if (tid == 0) sh.bk = -1;
  cta_sync<NT>();
  for (int i = tid; i < U; i += NT) {
    const int b = bin_of(cand[i]);
    atomicAdd(&cnt32[b >> 1], 1u << ((b & 1) * 16));
  }
  cta_sync<NT>();
  int own = 0;
#pragma unroll
  for (int j = 0; j < PB; ++j) own += static_cast<int>(cnt[tid * PB + j]);
  int tot;
  int st = Block<NT>::excl_scan_int(own, sh.sc.red_i, tot);
#pragma unroll
  for (int j = 0; j < PB; ++j) {
    const int b = tid * PB + j;
    const int cb = static_cast<int>(cnt[b]);
    fil[b] = static_cast<uint16_t>(st);
    if (cb > 0 && st < kk && kk <= st + cb) {
      sh.bk = b;
      sh.nk = st + cb;
    }
    st += cb;
  }
  cta_sync<NT>();
  const int bk = sh.bk, nk = sh.nk;  // bk >= 0: the bins hold U >= kk entries
  int g = 0;
#pragma unroll
  for (int j = 0; j < PB; ++j) {
    const int b = tid * PB + j;
    if (b <= bk) g = max(g, static_cast<int>(cnt[b]));
  }
  const int gmax = -Block<NT>::min_int(-g, sh.sc.red_i);
  if (U + nk > CAP || gmax > kMaxGroup) return 0;
  if constexpr (DT == 1) {  // float rows (bf16 rows reach this finish only as a rare fallback)
    if (!rc.capture && !rc.greedy && !rc.positional && !rc.minp_first &&
        U + bk + 1 + 2 * kMaxGroup + NT / 32 <= CAP) {  // uniform: only the token is wanted
      finish_unsorted<DT, NT, NB>(p, rc, cand, sh, U, m, Z, inv, kk, bk);
      return 1;
    }
  }

  // Placement of the bins up to bk behind the pool, then in-bin ranks into cand[0..nk).
  for (int i = tid; i < U; i += NT) {
    const uint64_t e = cand[i];
    const int b = bin_of(e);
    if (b <= bk) {
      const int sh16 = (b & 1) * 16;
      cand[U + static_cast<int>((atomicAdd(&fil32[b >> 1], 1u << sh16) >> sh16) & 0xFFFFu)] = e;
    }
  }
  cta_sync<NT>();
  for (int i = tid; i < nk; i += NT) {
    const uint64_t e = cand[U + i];
    const int b = bin_of(e);
    const int gb = static_cast<int>(cnt[b]);
    const int b0 = static_cast<int>(fil[b]) - gb;
    int r = 0;
    for (int j = b0; j < b0 + gb; ++j) r += cand[U + j] > e ? 1 : 0;
    cand[b0 + r] = e;
  }
  cta_sync<NT>();
  // K ends with the tie group of the kk-th largest.
  const uint32_t kth = ckey_key(cand[kk - 1]);
  int endv = nk;
  for (int b0 = kk; b0 < nk; b0 += NT) {  // uniform trip count
    const int i = b0 + tid;
    const uint32_t key = ckey_key(cand[min(i, nk - 1)]);
    if (i < nk && key != kth) endv = min(endv, i);
  }
  const int n = Block<NT>::min_int(endv, sh.sc.red_i);
  finish_sorted<DT, NT>(p, rc, cand, sh, n, m, Z);
  return 1;
}

// ------------------------------------------------------------------------------------------
// bf16 finish by exact-value bins, without sorting. Every candidate is >= tau, so its 16-bit key
// lies in [tau16, m16], m16 the row maximum's. A bin is one value, i.e. one tie group: bin d =
// m16 - key16 when that range has at most NB codes, else the dense rank of the value among the
// candidates' distinct values (a presence bitmap over the range and word prefix counts), stored
// in the key's low 16 bits (zero in bf16 keys, and equal for equal values, so every comparison of
// keys is unchanged). One exclusive scan over the bins of the counts and of the masses count_d
// 2^((x_d - m)c) gives all three cuts: a group leaves K when at least k tokens are larger, leaves
// P when the mass of the larger tokens exceeds top_p Z, leaves M when z - z_max < ln(min_p); each
// condition, once true, stays true for every later group, so S is the bins before the first
// excluded one. The pool holds the candidates in ascending id order; each warp places its part of
// it into its bins' slots in order (a stable counting sort), so S lands in canonical order.
// Warp w's part: pool[w capw, (w + 1) capw) within pool[0..U); work: WORK_BYTES of free shared
// memory.
// Returns false, having written no output, when this path does not apply (no sample threshold,
// more than NB distinct values, more members of S than the work area holds) or tau overshot the
// k-th largest.
// ------------------------------------------------------------------------------------------
// Which bins the bf16 finish uses for a row: none (ok false: no sample threshold, a float row or
// a code range beyond kBinsCodes), code distances from the maximum (R <= kBinsMax codes), or dense
// value ranks from a presence bitmap of nw words over the code range, set while the pool is
// gathered.
constexpr int kBinsMax = 1024;     // bins at most
constexpr int kBinsCodes = 65536;  // codes in [tau16, m16] at most
struct BinsPlan {
  bool ok, dense;
  int m16, R, nw;
  float tau_x;  // the value of the pool's key floor
};
__device__ __forceinline__ BinsPlan bins_plan(const RowCtx& rc, uint32_t tau, float m, bool bf16) {
  BinsPlan b;
  b.m16 = static_cast<int>(Keys<0>::key(m) >> 16);
  b.R = b.m16 - static_cast<int>(tau >> 16) + 1;
  b.ok = bf16 && rc.k_active && tau > kKeyLowestFinite && b.R >= 1 && b.R <= kBinsCodes;
  b.dense = b.ok && b.R > kBinsMax;
  b.nw = b.dense ? (b.R + 31) >> 5 : 0;
  b.tau_x = Keys<0>::value(tau);
  return b;
}

template <int NT, int WORK_BYTES, int BITW>
__device__ __noinline__ bool finish_bins(const Params& p, const RowCtx rc, uint64_t* pool, int capw, int U,
                                         Shared<NT>& sh, const BinsPlan bp, float m, float Z, unsigned char* work,
                                         uint32_t* bm) {
  using K = Keys<0>;
  constexpr int NW = NT / 32;
  constexpr int NB = kBinsMax;
  constexpr int BMW = kBinsCodes / 32;  // presence bitmap words at most
  // work: wc[NW][NB] (u16: per-warp counts, then per-warp slots) | start[NB] | mab[NB] |
  // code[NB] (u16) | tmp[] (S in canonical order). bm: the presence bitmap (BMW words), then
  // pre[BMW] (u16); tmp may overlap them, being written only after their last read.
  constexpr int OFF_START = NW * NB * 2;
  constexpr int OFF_MAB = OFF_START + NB * 4;
  constexpr int OFF_CODE = OFF_MAB + NB * 4;
  constexpr int OFF_TMP = OFF_CODE + NB * 2;
  constexpr int TMPCAP = (WORK_BYTES - OFF_TMP) / 8;  // placed entries at most
  static_assert(OFF_TMP % 16 == 0 && TMPCAP > 0 && BITW * 2 >= BMW * 3, "work area");
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int m16 = bp.m16, R = bp.R, nw = bp.nw;
  const bool dense = bp.dense;  // uniform
  uint16_t* wc = reinterpret_cast<uint16_t*>(work);
  uint32_t* start = reinterpret_cast<uint32_t*>(work + OFF_START);
  float* mab = reinterpret_cast<float*>(work + OFF_MAB);
  uint16_t* code = reinterpret_cast<uint16_t*>(work + OFF_CODE);
  uint64_t* tmp = reinterpret_cast<uint64_t*>(work + OFF_TMP);
  uint16_t* pre = reinterpret_cast<uint16_t*>(bm + BMW);
  int nb = R;  // bins in use
  int r = 0, w0 = 0, w1 = 0;
  if (dense) {
    // Dense ranks: the distinct values above a word, by a scan over runs of consecutive words.
    const int PWd = (nw + NT - 1) / NT;
    w0 = min(tid * PWd, nw);
    w1 = min(w0 + PWd, nw);
    int own = 0;
#pragma unroll 1
    for (int i = w0; i < w1; ++i) own += __popc(bm[i]);
    r = Block<NT>::excl_scan_int(own, sh.sc.red_i, nb);
    if (nb > NB) return false;  // uniform
  }
  {
    uint32_t* wc32 = reinterpret_cast<uint32_t*>(wc);
    const int half = (nb + 1) >> 1;  // counter words in use per warp
#pragma unroll 1
    for (int j = tid; j < half; j += NT) {
#pragma unroll
      for (int v = 0; v < NW; ++v) wc32[v * (NB / 2) + j] = 0;
    }
#pragma unroll 1
    for (int i = w0; i < w1; ++i) {
      pre[i] = static_cast<uint16_t>(r);
      r += __popc(bm[i]);
    }
  }
  cta_sync<NT>();
  // The bin of a candidate; in the dense case also recorded in its key's low 16 bits.
  auto bin_of = [&](uint64_t e) -> int {
    const uint32_t k = ckey_key(e);
    return dense ? static_cast<int>(k & 0xFFFFu) : m16 - static_cast<int>(k >> 16);
  };
  auto value_of = [&](int b) {
    const uint32_t c16 = dense ? static_cast<uint32_t>(code[b]) : static_cast<uint32_t>(m16 - b);
    return K::value(c16 << 16);
  };

  // Per-warp counts (16-bit, two to a word): warp w takes its part pool[q0, q1); in the dense case
  // each entry's bin goes into its key and each bin's value into code[].
  const int q0 = min(w * capw, U), q1 = min(q0 + capw, U);
  uint16_t* wcw = wc + w * NB;
  uint32_t* wcw32 = reinterpret_cast<uint32_t*>(wcw);
#pragma unroll 1
  for (int i = q0 + lane; i < q1; i += 32) {
    const uint64_t e = pool[i];
    const uint32_t c16 = ckey_key(e) >> 16;
    const int d = m16 - static_cast<int>(c16);
    int b = d;
    if (dense) {
      b = pre[d >> 5] + __popc(bm[d >> 5] & ((1u << (d & 31)) - 1u));
      pool[i] = e | (static_cast<uint64_t>(b) << 32);
      code[b] = static_cast<uint16_t>(c16);  // every writer stores the same value
    }
    atomicAdd(&wcw32[b >> 1], 1u << ((b & 1) * 16));
  }
  cta_sync<NT>();

  // Exclusive scans of counts and masses over the bins; thread t owns a run of consecutive bins.
  const int PBk = (nb + NT - 1) / NT;
  const int b0 = min(tid * PBk, nb), b1 = min(b0 + PBk, nb);
  int c_own = 0;
  float w_own = 0.f, wM_own = 0.f;
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    int cb = 0;
#pragma unroll
    for (int v = 0; v < NW; ++v) cb += wc[v * NB + b];
    c_own += cb;
    const float wb = cb > 0 ? static_cast<float>(cb) * ex2_approx((value_of(b) - m) * rc.c) : 0.f;
    w_own += wb;
    if (zrel_of(value_of(b), m, rc.invT) >= rc.ln_min_p) wM_own += wb;
  }
  int c_tot;
  float w_tot;
  int c = c_own;
  float wm = w_own;
  Block<NT>::excl_scan2(c, wm, sh.sc.red_i, sh.sc.red_f, c_tot, w_tot);
  if (c_tot < rc.k) return false;  // uniform: tau overshot
  float ZP = Z;  // the mass top-p measures against
  if (rc.minp_first) {  // uniform: M's mass, when M lies inside the pool (its floor fails min-p)
    if (!(zrel_of(bp.tau_x, m, rc.invT) < rc.ln_min_p)) return false;
    ZP = Block<NT>::sum(wM_own, sh.sc.red_f);
  }
  const float thr = rc.top_p * ZP;
  int cut = nb;
  int npos = c_tot;  // positional: the support's length (the first position any truncation removes)
#pragma unroll 1
  for (int b = b0; b < b1; ++b) {
    int cb = 0;
#pragma unroll
    for (int v = 0; v < NW; ++v) {  // counts become the warps' first slots in the bin
      const int t = wc[v * NB + b];
      wc[v * NB + b] = static_cast<uint16_t>(c + cb);
      cb += t;
    }
    start[b] = static_cast<uint32_t>(c);
    mab[b] = wm;
    const float wb = cb > 0 ? ex2_approx((value_of(b) - m) * rc.c) : 0.f;  // one member's weight
    const bool out_m = rc.m_active && cb > 0 && zrel_of(value_of(b), m, rc.invT) < rc.ln_min_p;
    if (cb > 0 && cut == nb) {
      const bool out_k = c >= rc.k;
      const bool out_p = rc.p_active && wm > thr;
      if (out_k || out_p || out_m) cut = b;
    }
    if (rc.positional && cb > 0) {  // the first position in this bin that a truncation removes
      if (rc.k_active && c + cb > rc.k) npos = min(npos, rc.k);
      if (rc.p_active && wm + static_cast<float>(cb - 1) * wb > thr) {  // member j's mass before: wm + j wb
        const float q = (thr - wm) / wb;
        const int j = wm > thr ? 0 : (q >= static_cast<float>(cb) ? cb : static_cast<int>(floorf(q)) + 1);
        npos = min(npos, c + j);
      }
      if (out_m) npos = min(npos, c);
    }
    c += cb;
    wm += static_cast<float>(cb) * wb;
  }
  cut = Block<NT>::min_int(cut, sh.sc.red_i);  // its barriers publish start[], mab[] and the slots
  int nS = cut < nb ? static_cast<int>(start[cut]) : c_tot;  // >= 1: the top group always passes
  float ZS = cut < nb ? mab[cut] : w_tot;
  if (rc.positional) {  // S: the first npos positions; place every bin up to the one holding the last
    npos = Block<NT>::min_int(npos, sh.sc.red_i);
    int lo = 0, hi = nb - 1;  // the last bin starting at or before position npos - 1
#pragma unroll 1
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<int>(start[mid]) <= npos - 1) lo = mid;
      else hi = mid - 1;
    }
    ZS = mab[lo] + static_cast<float>(npos - static_cast<int>(start[lo])) * ex2_approx((value_of(lo) - m) * rc.c);
    cut = lo + 1;
    nS = npos;
  }
  const int n_place = cut < nb ? static_cast<int>(start[cut]) : c_tot;
  if (n_place > TMPCAP) return false;  // uniform
  const float logZS = logf(ZS);

  // Stable placement of S: each warp walks its part of the pool in order, 32 entries at a time
  // (two tiles per round, whose ballots overlap); a lane's peers (the lanes of the tile with its
  // bin) come from one ballot per bin bit.
  const int nbits = 32 - __clz(max(nb - 1, 1));
  auto place_tile = [&](uint64_t e, int b, unsigned peers, bool valid) {
    const bool in_s = valid && b < cut;
    int slot = 0;
    if (in_s) {
      slot = wcw[b];
      tmp[slot + __popc(peers & ((1u << lane) - 1u))] = e;
    }
    __syncwarp();
    if (in_s && lane == __ffs(static_cast<int>(peers)) - 1) wcw[b] = static_cast<uint16_t>(slot + __popc(peers));
    __syncwarp();
  };
  if (q1 - q0 <= 32) {  // warp-uniform: one tile
    const int ia = q0 + lane;
    const bool va = ia < q1;
    const uint64_t ea = va ? pool[ia] : 0;
    const int ba = va ? bin_of(ea) : 0;
    unsigned pa = __ballot_sync(kFull, va);
#pragma unroll 1
    for (int k = 0; k < nbits; ++k) {
      const bool xa = (ba >> k) & 1;
      const unsigned la = __ballot_sync(kFull, xa);
      pa &= xa ? la : ~la;
    }
    if (q0 < q1) place_tile(ea, ba, pa, va);  // warp-uniform
  } else {
#pragma unroll 1
  for (int i0 = q0; i0 < q1; i0 += 64) {  // warp-uniform
    const int ia = i0 + lane, ib = ia + 32;
    const bool va = ia < q1, vb = ib < q1;
    const uint64_t ea = va ? pool[ia] : 0, eb = vb ? pool[ib] : 0;
    const int ba = va ? bin_of(ea) : 0, bb = vb ? bin_of(eb) : 0;
    unsigned pa = __ballot_sync(kFull, va), pb = __ballot_sync(kFull, vb);
#pragma unroll 1
    for (int k = 0; k < nbits; ++k) {
      const bool xa = (ba >> k) & 1, xb = (bb >> k) & 1;
      const unsigned la = __ballot_sync(kFull, xa), lb = __ballot_sync(kFull, xb);
      pa &= xa ? la : ~la;
      pb &= xb ? lb : ~lb;
    }
    place_tile(ea, ba, pa, va);
    if (i0 + 32 < q1) place_tile(eb, bb, pb, vb);  // warp-uniform
  }
  }
  cta_sync<NT>();

  if (rc.greedy) {  // tmp[0]: the lowest id of the largest value
    if (tid == 0) write_greedy_row(p, rc.row, rc.capture, ckey_id(tmp[0]));
    return true;
  }

  // Exponential race over S, spread evenly over the threads; capturing rows also write the first
  // n_out members, tmp being in canonical order.
  const int n_out = rc.capture ? min(nS, p.W) : 0;
  int32_t* ids = p.support_ids + static_cast<int64_t>(rc.row) * p.W;
  float* lps = (rc.capture && p.support_logprobs) ? p.support_logprobs + static_cast<int64_t>(rc.row) * p.W : nullptr;
  float best = -INFINITY, bx = 0.f;
  uint32_t bid = 0xFFFFFFFFu;
#pragma unroll 1
  for (int i = tid; i < nS; i += NT) {
    const uint64_t e = tmp[i];
    const float x = K::value(ckey_key(e));
    const uint32_t id = ckey_id(e);
    const float zr = zrel_of(x, m, rc.invT);
    const float sc = race_member_score(p.seed, p.step, rc.noise_row, id, zr);
    if (race_better(sc, id, best, bid)) { best = sc; bid = id; bx = x; }
    if (i < n_out) {
      ids[i] = static_cast<int32_t>(id);
      if (lps) lps[i] = zr - logZS;
    }
  }
  Block<NT>::race_argmax(best, bid, bx, sh.sc.red_f, sh.sc.red_u, sh.sc.red_x);
  if (tid == 0) {
    p.tokens[rc.row] = static_cast<int32_t>(bid);
    if (rc.capture) {
      p.lengths[rc.row] = nS;
      p.row_status[rc.row] = nS > p.W ? 1 : 0;
      p.selected_logprob[rc.row] = zrel_of(bx, m, rc.invT) - logZS;
    } else {
      p.row_status[rc.row] = 0;
      if (p.lengths) p.lengths[rc.row] = 0;
    }
  }
  if (rc.capture && p.support_mask && nS > p.W) write_support_mask_ids<NT>(p, rc, tmp, nS);  // uniform
  return true;
}

// ------------------------------------------------------------------------------------------
// Finish of the row: the bucket finish, else the select-and-sort finish, else the multi-pass path.
// area[0..AREA) is the ring's space followed by the candidate buffer, all free again; the
// candidates have been gathered into area[0..U).
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int AREA>
__device__ __noinline__ void finish_row(const Params& p, const RowCtx rc, uint64_t* area, int U, bool complete,
                                        Shared<NT>& sh, uint32_t tau) {
  using K = Keys<DT>;
  const int tid = threadIdx.x;
  const float m = sh.row_m, Z = sh.row_Z;
  // NaN (poisons the sum), +inf (becomes the maximum) or no finite logit at all.
  if (!(m > -INFINITY && m < INFINITY) || !(Z == Z)) {
    if (tid == 0) write_bad_row(p, rc.row, rc.capture);
    return;
  }
  // In the min-p-first order top-p measures against M's mass: from the pool when M lies inside it
  // (the pool is every finite token, or its floor fails min-p), else on the multi-pass path.
  const bool m_in_pool = !rc.minp_first || tau <= kKeyLowestFinite || zrel_of(K::value(tau), m, rc.invT) < rc.ln_min_p;
  if (complete && U >= 1 && m_in_pool) {
    // lo: the low end of the bucket finish's value range. Every candidate is >= tau, so tau's value
    // serves when tau is a threshold; else (every finite token is a candidate), and in the min-p-first
    // order, which needs M's mass among the candidates anyway, the smallest candidate.
    float lo = K::value(tau);
    float ZP = Z;  // the mass top-p measures against
    if (tau <= kKeyLowestFinite || rc.minp_first) {  // uniform
      lo = INFINITY;
      float zm = 0.f;  // M's mass among the candidates
      for (int i = tid; i < U; i += NT) {
        const float x = K::value(ckey_key(area[i]));
        lo = fminf(lo, x);
        if (rc.minp_first && zrel_of(x, m, rc.invT) >= rc.ln_min_p) zm += ex2_approx((x - m) * rc.c);
      }
      lo = Block<NT>::min_f(lo, sh.sc.red_f);
      if (rc.minp_first) ZP = Block<NT>::sum(zm, sh.sc.red_f);
    }
    const int r = finish_bucket<DT, NT, AREA>(p, rc, area, sh, U, m, ZP, lo, tau);
    if (r > 0) return;
    if (r == 0 && finish_fast<DT, NT, AREA>(p, rc, area, sh, U, m, ZP, tau)) return;
    cta_sync<NT>();
  }
  general_path<DT, NT, AREA>(p, rc, area, sh, m, Z);
}

// ------------------------------------------------------------------------------------------
// The marked vectors, ascending, from the candidate bitmap into list[0..marked) (written only if
// marked <= LIST): thread t takes a run of bitmap words, a block scan places its vectors. Each word
// is cleared once read, so that the bitmap's space starts the bins finish's presence bitmap (whose
// words past the pass's are cleared here too when the plan is dense). Returns marked; the list is
// complete on return.
// ------------------------------------------------------------------------------------------
template <int NT, int SB, int LIST, typename ST>
__device__ __forceinline__ int build_list(const ST& st, uint32_t* bitmap, uint32_t* list, const BinsPlan& bins,
                                          Shared<NT>& sh) {
  const int tid = threadIdx.x;
  const int nwords = st.bits_ok ? st.nchunks * (SB / 16 / 32) : 0;
  const int per = (nwords + NT - 1) / NT;
  const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
  int mine = 0;
#pragma unroll 1
  for (int w = w0; w < w1; ++w) mine += __popc(bitmap[w]);
  int marked;
  int off = Block<NT>::excl_scan_int(mine, sh.sc.red_i, marked);
  if (marked <= LIST) {  // uniform
#pragma unroll 1
    for (int w = w0; w < w1; ++w) {
      uint32_t b = bitmap[w];
      bitmap[w] = 0;
#pragma unroll 1
      while (b) {
        const int i = __ffs(static_cast<int>(b)) - 1;
        b &= b - 1;
        list[off++] = static_cast<uint32_t>(w * 32 + i);
      }
    }
    if (bins.dense)
#pragma unroll 1
      for (int w = nwords + tid; w < bins.nw; w += NT) bitmap[w] = 0;
  }
  cta_sync<NT>();
  return marked;
}

// ------------------------------------------------------------------------------------------
// The candidates into pool[0..U) in no particular order, for rows whose finish sorts the full keys
// (float rows: the bucket and select-and-sort finishes): one sweep, thread t reading list entries
// t, t + NT, ... (RV rounds of loads in flight), a warp-aggregated reservation per batch. Returns U,
// or -1 past POOL entries.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int RV, int POOL, typename ST>
__device__ __forceinline__ int gather_pool_unordered(const ST& st, const uint32_t* list, int marked, uint64_t* pool,
                                                    Shared<NT>& sh) {
  using E = Elem<DT>;
  using K = Keys<DT>;
  constexpr int VEC = E::kVec;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) sh.pool_n = 0;
  cta_sync<NT>();
  const int nr = (marked + NT - 1) / NT;
#pragma unroll 1
  for (int r0 = 0; r0 < nr; r0 += RV) {  // uniform
    uint4 v[RV];
    uint32_t mask[RV];
    uint32_t vi[RV];
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      const int i = (r0 + j) * NT + tid;
      mask[j] = 0;
      vi[j] = 0;
      if (i < marked) {
        vi[j] = list[i];
        v[j] = ld_once(st.body + vi[j]);
      }
    }
    int n = 0;
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      if ((r0 + j) * NT + tid < marked) mask[j] = E::ge_mask(v[j], st.tau_f);
      n += __popc(mask[j]);
    }
    const int incl = warp_incl_scan(n);
    int base = 0;
    if (lane == 31 && incl > 0) base = atomicAdd(&sh.pool_n, incl);
    int at = __shfl_sync(kFull, base, 31) + incl - n;
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      const uint32_t id0 = st.head + vi[j] * VEC;
      uint32_t mk = mask[j];
#pragma unroll 1
      while (mk) {
        const int e = __ffs(static_cast<int>(mk)) - 1;
        mk &= mk - 1;
        if (at < POOL) pool[at] = make_ckey(K::key(E::get_dyn(v[j], e)), id0 + static_cast<uint32_t>(e));
        ++at;
      }
    }
  }
  const int n_ext = sh.n_ext;
  if (tid < n_ext) {
    const int at = atomicAdd(&sh.pool_n, 1);
    if (at < POOL) pool[at] = sh.ext[tid];
  }
  cta_sync<NT>();
  const int U = sh.pool_n;
  return U <= POOL ? U : -1;
}

// ------------------------------------------------------------------------------------------
// The candidates into pool[0..U) in ascending id order: the head scalars, the marked vectors
// list[0..marked) (read again from L2), the tail scalars. Thread t takes a run of `per`
// consecutive marked vectors, RV at a time: kept in registers when the run fits in one batch,
// else counted in one sweep and read again in a second. Dense bins plans also get each
// candidate's bit in the presence bitmap. Returns U, or -1 (nothing usable) past POOL entries.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int RV, int POOL, typename ST>
__device__ __forceinline__ int gather_pool(const ST& st, const uint32_t* list, int marked, int per, uint64_t* pool,
                                           Shared<NT>& sh, const BinsPlan& bins, uint32_t* bitmap) {
  using E = Elem<DT>;
  using K = Keys<DT>;
  constexpr int VEC = E::kVec;
  const int tid = threadIdx.x;
  const int n_ext = sh.n_ext;
  const int i0 = min(tid * per, marked), i1 = min(i0 + per, marked);
  uint4 v[RV];
  uint32_t mask[RV];
  auto load = [&](int j0) {  // every load of the batch is issued before any result is used
#pragma unroll
    for (int j = 0; j < RV; ++j)
      if (j0 + j < i1) v[j] = ld_once(st.body + list[j0 + j]);
#pragma unroll
    for (int j = 0; j < RV; ++j) mask[j] = (j0 + j < i1) ? E::ge_mask(v[j], st.tau_f) : 0u;
  };
  auto mark_present = [&](uint32_t key) {  // the value's presence bit
    if (bins.dense) {
      const int d = bins.m16 - static_cast<int>(key >> 16);
      const uint32_t bit = 1u << (d & 31);
      atomicOr(&bitmap[d >> 5], bit);  // result unused: the loop does not wait for it
    }
  };
  auto store = [&](int j0, int& at) {
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      if (j0 + j < i1) {
        const uint32_t id0 = st.head + list[j0 + j] * VEC;
        uint32_t mk = mask[j];
#pragma unroll 1
        while (mk) {
          const int e = __ffs(static_cast<int>(mk)) - 1;
          mk &= mk - 1;
          const uint32_t key = K::key(E::get_dyn(v[j], e));
          pool[at++] = make_ckey(key, id0 + static_cast<uint32_t>(e));
          mark_present(key);
        }
      }
    }
  };
  int n = 0;
#pragma unroll 1
  for (int j0 = i0; j0 < i1; j0 += RV) {
    load(j0);
#pragma unroll
    for (int j = 0; j < RV; ++j) n += __popc(mask[j]);
  }
  int n_body;
  int at = Block<NT>::excl_scan_int(n, sh.sc.red_i, n_body);
  if (n_body + n_ext > POOL) return -1;  // uniform
  // the head scalars come first (ids below the body's), the tail scalars last
  int n_head = 0, rank = 0;
  const uint64_t xe = tid < n_ext ? sh.ext[tid] : 0;
#pragma unroll 1
  for (int j = 0; j < n_ext; ++j) {
    const uint32_t idj = ckey_id(sh.ext[j]);
    n_head += idj < st.head ? 1 : 0;
    rank += (tid < n_ext && idj < ckey_id(xe)) ? 1 : 0;
  }
  at += n_head;
  if (per > RV) {  // uniform
#pragma unroll 1
    for (int j0 = i0; j0 < i1; j0 += RV) {
      load(j0);
      store(j0, at);
    }
  } else if (i0 < i1) {
    store(i0, at);
  }
  if (tid < n_ext) {
    pool[ckey_id(xe) < st.head ? rank : n_body + rank] = xe;
    mark_present(ckey_key(xe));
  }
  return n_body + n_ext;
}

// ------------------------------------------------------------------------------------------
// The candidates >= tau of a row's slice pools (in the workspace, slices s0 .. s0 + SL - 1 with
// sh.sx_U[c] entries each), concatenated in slice order, into pool[0..total): thread t takes a run
// of `per` consecutive entries of the concatenation, RV at a time (kept in registers when the run
// fits in one batch, else counted in one sweep and read again in a second), and one block scan
// places them. Reads bypass L1 (the pools were written by other CTAs). Returns total, or -1 past
// POOL entries.
// ------------------------------------------------------------------------------------------
template <int NT, int RV, int POOL>
__device__ __noinline__ int merge_slice_pools(const Params& p, int64_t s0, int SL, int N, uint32_t tau,
                                              uint64_t* pool, Shared<NT>& sh) {
  const int tid = threadIdx.x;
  const int per = (N + NT - 1) / NT;
  const int i0 = min(tid * per, N), i1 = min(i0 + per, N);
  const uint64_t* base = p.slice_pool + s0 * p.slice_cap;
  auto at = [&](int i) {  // entry i of the concatenation
    int c = 0;
#pragma unroll 1
    while (c < SL - 1 && i >= sh.sx_U[c]) {
      i -= sh.sx_U[c];
      ++c;
    }
    return base + static_cast<int64_t>(c) * p.slice_cap + i;
  };
  uint64_t v[RV];
  uint32_t keep = 0;
  auto load = [&](int j0) {
    keep = 0;
#pragma unroll
    for (int j = 0; j < RV; ++j) {
      if (j0 + j < i1) {
        v[j] = __ldcg(reinterpret_cast<const unsigned long long*>(at(j0 + j)));
        keep |= static_cast<uint32_t>(ckey_key(v[j]) >= tau) << j;
      }
    }
  };
  int n = 0;
#pragma unroll 1
  for (int j0 = i0; j0 < i1; j0 += RV) {
    load(j0);
    n += __popc(keep);
  }
  int total;
  int o = Block<NT>::excl_scan_int(n, sh.sc.red_i, total);
  if (total > POOL) return -1;  // uniform
  auto store = [&]() {
#pragma unroll
    for (int j = 0; j < RV; ++j)
      if ((keep >> j) & 1u) pool[o++] = v[j];
  };
  if (per > RV) {  // uniform
#pragma unroll 1
    for (int j0 = i0; j0 < i1; j0 += RV) {
      load(j0);
      store();
    }
  } else {
    store();  // the run is still in registers
  }
  cta_sync<NT>();
  return total;
}

// Zero the N entries that a row's slices published (the concatenation of their pools, sh.sx_U[c]
// entries each, negative counts meaning none), after merge_slice_pools has read them.
template <int NT>
__device__ __noinline__ void clear_slice_pools(const Params& p, int64_t s0, int SL, int N, Shared<NT>& sh) {
  uint64_t* base = p.slice_pool + s0 * p.slice_cap;
#pragma unroll 1
  for (int i = threadIdx.x; i < N; i += NT) {
    int c = 0, j = i;
#pragma unroll 1
    while (c < SL - 1 && j >= max(sh.sx_U[c], 0)) {
      j -= max(sh.sx_U[c], 0);
      ++c;
    }
    base[static_cast<int64_t>(c) * p.slice_cap + j] = 0ull;
  }
}

// ------------------------------------------------------------------------------------------
// The kernel: one CTA per row.
// ------------------------------------------------------------------------------------------
template <int DT, int NT, int NS, int SB, int BITW, int MINB, int GSN>
__global__ void __launch_bounds__(NT, MINB) fused_kernel(const __grid_constant__ Params p) {
  using E = Elem<DT>;
  using K = Keys<DT>;
  constexpr int VEC = E::kVec;
  // Dynamic shared memory: the ring (NS * SB bytes), then the bitmap (BITW words). After the pass
  // the ring's space holds the candidate pool (POOL entries: half of it, five eighths for the
  // deep rings of the wide class) and then the list of marked vectors; everything past the pool is
  // the finishes' work space, except the last SCR bytes (inside the bitmap, read out by then): the
  // warp histograms and mass bins of the sorting and multi-pass finishes.
  constexpr int DYN = NS * SB + BITW * 4;
  constexpr int POOL = (NS * SB / 8) * (NS >= 8 ? 5 : 4) / 8;
  constexpr int LIST = (NS * SB - POOL * 8) / 4;  // marked vectors at most (4-byte indices)
  constexpr int SCR = (NT / 32) * 256 * 4 + 256 * 8;
  constexpr int AREA = (DYN - SCR) / 8;  // 8-byte entries of the finishes' space
  static_assert((NS * SB) % 32 == 0 && BITW * 4 >= SCR && DYN % 8 == 0 && SCR % 8 == 0, "layout");
  extern __shared__ __align__(128) unsigned char dyn_smem[];
  unsigned char* ring = dyn_smem;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn_smem + NS * SB);
  __shared__ Shared<NT> sh;
  __shared__ uint64_t bars[NS];  // stage filled

  const int C = p.split;    // CTAs per row as a cluster (distributed shared memory)
  const int SL = p.slices;  // CTAs per row meeting through the workspace (at most one of C, SL is > 1)
  const int NP = C * SL;    // CTAs (slices) per row
  const int row = static_cast<int>(blockIdx.x) / NP;
  const int crank = static_cast<int>(blockIdx.x) % NP;  // this CTA's slice of the row
  const int tid = threadIdx.x;

  // ---- the row's place and this CTA's slice of it: from the kernel arguments alone ----
  RowCtx rc;
  rc.row = row;
  rc.noise_row = static_cast<uint32_t>(p.row_offset + row);
  rc.V = p.V;
  rc.rowp = static_cast<const unsigned char*>(p.logits) + static_cast<int64_t>(row) * p.row_stride * E::kBytes;
  rc.head = static_cast<int64_t>((16u - (reinterpret_cast<uintptr_t>(rc.rowp) & 15u)) & 15u) / E::kBytes;
  if (rc.head > rc.V) rc.head = rc.V;
  rc.nvec = (rc.V - rc.head) / VEC;
  rc.body_end = rc.head + rc.nvec * VEC;
  // This CTA's slice of the vectors; the first slice also reads the head scalars, the last the tail.
  rc.vec0 = rc.nvec * crank / NP;
  rc.svec = rc.nvec * (crank + 1) / NP - rc.vec0;
  rc.x_head = crank == 0 ? static_cast<int>(rc.head) : 0;
  rc.x_tail = crank == NP - 1 ? static_cast<int>(rc.V - rc.body_end) : 0;

  // ---- the first ring stages go out before anything is loaded: the row's first bytes travel while
  // its parameters load ----
  Streamer<DT, NT, NS, SB, BITW, GSN> st(sh, ring, bars, bitmap, rc);
  st.stalled = (p.flags & kFlagTestStall) != 0;
  const int early = min(NS, st.nchunks);
  if (tid == 0) {
    sh.sc.whist = reinterpret_cast<uint32_t*>(dyn_smem + DYN - SCR);
    sh.mass = reinterpret_cast<unsigned long long*>(dyn_smem + DYN - 256 * 8);
    sh.n_ext = 0;
    sh.timed_out = 0;
    sh.samp_d = -1;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars[s], 1);  // the issuer's arrive; the copy's bytes complete it
      sh.left[s] = 0;
    }
    mbar_init_fence();
    for (int s = 0; s < early; ++s)
      if (!(st.stalled && s == 0)) st.issue(s, s);
    sh.issued = early;
  }

  // ---- the row's parameters ----
  rc.T = p.temperature[row];
  rc.k = p.top_k[row];
  rc.top_p = p.top_p[row];
  float min_p = p.min_p[row];
  rc.capture = p.capture_rows != nullptr && p.capture_rows[row] != 0;
  rc.greedy = (p.flags & kFlagGreedyT0) != 0 && rc.T == 0.f;
  rc.positional = (p.flags & kFlagPositional) != 0;
  if (rc.greedy) {  // the largest tie group is found as a top-1 support; its lowest id is the token
    rc.T = 1.f;
    rc.k = 1;
    rc.top_p = 1.f;
    min_p = 0.f;
  }
  const bool params_ok = (rc.T > 0.f) && (rc.T < INFINITY) && (rc.top_p >= 0.f) && (min_p >= 0.f) && (min_p <= 1.f);
  if (!params_ok) {  // uniform: every thread read the same parameters
    if (tid == 0) {
      st.drain();  // the early stages land before the CTA leaves
      write_bad_row(p, row, rc.capture);
    }
    return;
  }
  rc.c = kLog2e / rc.T;
  rc.invT = 1.f / rc.T;
  rc.k_active = rc.k >= 1 && static_cast<int64_t>(rc.k) < rc.V;
  rc.p_active = rc.top_p < 1.f;
  rc.m_active = min_p > 0.f;
  rc.ln_min_p = rc.m_active ? logf(min_p) : -INFINITY;
  rc.minp_first = (p.flags & kFlagMinPFirst) != 0 && rc.m_active && rc.p_active;  // else the same sets
  // Every row keeps the whole ring in flight. (Giving rows with long finishes a deeper ring than the
  // others, so that their passes end first, measured no faster on the mixed-k workloads.)
  st.begin(rc, NS, st.stalled ? kStallPolls : kWaitPolls);
  cta_sync<NT>();  // the barriers are initialised and the shared state is set

  // ---- the pass over the row ----
  st.fold_extra();
  st.stream();
  cta_sync<NT>();
  if (sh.timed_out) {  // not expected: a copy never completed. Leave nothing in flight, report the row.
    if (tid == 0) st.drain();
    if (NP == 1) {  // (a slice of a split row reports through the CTA that finishes the row)
      if (tid == 0) {
        p.tokens[row] = -1;
        p.row_status[row] = kRowTimeout;
        if (p.lengths) p.lengths[row] = 0;
      }
      return;
    }
  }

  // Softmax statistics of the row, in a fixed order.
  {
    // The warp's maximum, each thread's sum rescaled to it once, the warp's sum (xor butterflies give
    // every lane the same bits); then the warps' (max, sum) pairs merged in warp order.
    float m = st.m_t;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmax_nan(m, __shfl_xor_sync(kFull, m, o));
    float sm = st.m_t > -INFINITY ? st.s_t * ex2_approx((st.m_t - m) * rc.c) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFull, sm, o);
    if ((tid & 31) == 0) {
      sh.sc.red_f[tid >> 5] = m;
      sh.sc.red_x[tid >> 5] = sm;
    }
    cta_sync<NT>();
    constexpr int NW = NT / 32;
    m = sh.sc.red_f[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) m = fmax_nan(m, sh.sc.red_f[w]);
    sm = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = sh.sc.red_f[w];
      sm += mw > -INFINITY ? sh.sc.red_x[w] * ex2_approx((mw - m) * rc.c) : 0.f;
    }
    if (tid == 0) {
      sh.row_m = m;
      sh.row_Z = sm;
    }
    st.m_t = m;
    st.s_t = sm;
  }
  const float m = st.m_t, Z = st.s_t;
  uint64_t* pool = reinterpret_cast<uint64_t*>(ring);
  uint32_t* list = reinterpret_cast<uint32_t*>(ring + POOL * 8);  // marked vector indices, ascending
  constexpr int NW = NT / 32;

  if (SL > 1) {
    // ==== a row split into SL slices, ordinary CTAs that meet through the workspace ====
    // Each slice streams its part of the row, keeps its candidates (its logits >= its own sample
    // threshold) and publishes them with its threshold and statistics; the slice that arrives last
    // (one atomic ticket per row: no CTA ever waits for another) merges them in slice order and
    // finishes the row. While it does, the CTA slots of the other slices stream other rows.
    int U = -2;  // this slice's candidates; -1: more than fit, -2: a wait gave up
    if (!sh.timed_out) {  // uniform
      const BinsPlan no_bins = bins_plan(rc, kKeyLowestFinite, m, false);  // no presence bits here
      const int marked = build_list<NT, SB, LIST>(st, bitmap, list, no_bins, sh);
      U = -1;
      if (st.bits_ok && marked <= LIST) {  // uniform
        const int per = (marked + NT - 1) / NT;
        if (DT == 1)  // float rows are finished by sorting full keys: any pool order does
          U = gather_pool_unordered<DT, NT, 8, POOL>(st, list, marked, pool, sh);
        else
          U = per <= 2 ? gather_pool<DT, NT, 2, POOL>(st, list, marked, per, pool, sh, no_bins, bitmap)
                       : gather_pool<DT, NT, 8, POOL>(st, list, marked, per, pool, sh, no_bins, bitmap);
        if (U > p.slice_cap) U = -1;
      }
    }
    cta_sync<NT>();  // the pool is complete
    const int64_t s0 = static_cast<int64_t>(row) * SL;
    uint64_t* gpool = p.slice_pool + (s0 + crank) * p.slice_cap;
    for (int i = tid; i < U; i += NT) gpool[i] = pool[i];
    if (tid == 0) p.slice_rec[s0 + crank] = make_uint4(st.tau, __float_as_uint(m), __float_as_uint(Z), static_cast<uint32_t>(U));
    __threadfence();  // this slice's record and pool are visible device-wide before its ticket
    cta_sync<NT>();
    if (tid == 0) {
      const uint32_t prev = atomicAdd(&p.tickets[row], 1u);
      const int last = prev == static_cast<uint32_t>(SL - 1);
      if (last) p.tickets[row] = 0u;  // every slice has arrived: zero again for the next call
      __threadfence();  // the other slices' records and pools are read after their tickets
      sh.last = last;
    }
    cta_sync<NT>();
    if (!sh.last) return;

    // ---- the last slice to arrive finishes the row ----
    if (tid < SL) {
      const uint4 r = __ldcg(p.slice_rec + s0 + tid);
      sh.sx_tau[tid] = r.x;
      sh.sx_m[tid] = __uint_as_float(r.y);
      sh.sx_Z[tid] = __uint_as_float(r.z);
      sh.sx_U[tid] = static_cast<int>(r.w);
    }
    cta_sync<NT>();
    // The largest slice threshold: every slice holds all its logits >= its own threshold, so the
    // candidates >= tau_max of all slices are all the row's logits >= tau_max.
    uint32_t tau_max = 0;
    int worst = 0, N = 0;  // worst: -1 a slice's candidates did not fit, -2 a slice's wait gave up
    float m_all = -INFINITY, Z_all = 0.f;
    for (int c = 0; c < SL; ++c) {
      tau_max = max(tau_max, sh.sx_tau[c]);
      worst = min(worst, min(sh.sx_U[c], 0));
      N += max(sh.sx_U[c], 0);
      stat_merge(m_all, Z_all, sh.sx_m[c], sh.sx_Z[c], rc.c);  // slice order: the same bits every time
    }
    // The slices' candidates >= tau_max, concatenated in slice order (so in ascending id order).
    const int total = worst == 0 ? merge_slice_pools<NT, 8, POOL>(p, s0, SL, N, tau_max, pool, sh) : -1;
    const bool complete = total >= 0;
    // Every workspace byte this row's slices wrote goes back to zero (its ticket already has), so the
    // next call finds the workspace as the first one did, whatever its batch size or slice count.
    clear_slice_pools<NT>(p, s0, SL, N, sh);
    if (tid < SL) p.slice_rec[s0 + tid] = make_uint4(0u, 0u, 0u, 0u);
    if (worst == -2) {
      if (tid == 0) {
        p.tokens[row] = -1;
        p.row_status[row] = kRowTimeout;
        if (p.lengths) p.lengths[row] = 0;
      }
      return;
    }
    if (!(m_all > -INFINITY && m_all < INFINITY) || !(Z_all == Z_all)) {
      if (tid == 0) write_bad_row(p, row, rc.capture);
      return;
    }
    if (tid == 0) {
      sh.row_m = m_all;
      sh.row_Z = Z_all;
    }
    const BinsPlan bins = bins_plan(rc, tau_max, m_all, DT == 0);
    if (complete && bins.dense) {  // uniform: the presence bits of the merged candidates
      for (int i = tid; i < bins.nw; i += NT) bitmap[i] = 0;
      cta_sync<NT>();
      for (int i = tid; i < total; i += NT) {
        const int d = bins.m16 - static_cast<int>(ckey_key(pool[i]) >> 16);
        atomicOr(&bitmap[d >> 5], 1u << (d & 31));
      }
    }
    cta_sync<NT>();  // also publishes sh.row_m / sh.row_Z
    if (DT == 0 && complete && bins.ok) {
      const int Q = (total + NW - 1) / NW;
      if (finish_bins<NT, DYN - POOL * 8, BITW>(p, rc, pool, Q, total, sh, bins, m_all, Z_all, ring + POOL * 8, bitmap))
        return;
    }
    finish_row<DT, NT, AREA>(p, rc, pool, complete ? total : 0, complete, sh, tau_max);
    return;
  }

  if (C > 1) {
    // ==== a row split over a cluster of C CTAs (slices in id order) ====
    // Every CTA runs exactly the three cluster barriers below: nothing returns before the third.
    const BinsPlan no_bins = bins_plan(rc, kKeyLowestFinite, m, false);  // no presence bits here
    int U = -2;
    if (!sh.timed_out) {  // uniform
      const int marked = build_list<NT, SB, LIST>(st, bitmap, list, no_bins, sh);
      U = -1;
      if (st.bits_ok && marked <= LIST) {  // uniform
        const int per = (marked + NT - 1) / NT;
        U = per <= 2 ? gather_pool<DT, NT, 2, POOL>(st, list, marked, per, pool, sh, no_bins, bitmap)
                     : gather_pool<DT, NT, 8, POOL>(st, list, marked, per, pool, sh, no_bins, bitmap);
      }
    }
    if (tid < C) {  // this slice's entry into CTA tid's tables
      dsmem_st32(dsmem_addr(&sh.sx_tau[crank], tid), st.tau);
      dsmem_st32(dsmem_addr(&sh.sx_m[crank], tid), __float_as_uint(m));
      dsmem_st32(dsmem_addr(&sh.sx_Z[crank], tid), __float_as_uint(Z));
      dsmem_st32(dsmem_addr(&sh.sx_U[crank], tid), static_cast<uint32_t>(U));
    }
    cta_sync<NT>();  // the pool is complete
    cluster_sync_all();  // (1) every slice's threshold, statistics and pool size are published
    // The largest slice threshold: every slice holds all its logits >= its own threshold, so the
    // candidates >= tau_max of all slices are all the row's logits >= tau_max.
    uint32_t tau_max = 0;
    int worst = 0;  // -1: a slice incomplete, -2: a slice's wait gave up
    for (int c = 0; c < C; ++c) {
      tau_max = max(tau_max, sh.sx_tau[c]);
      worst = min(worst, min(sh.sx_U[c], 0));
    }
    // Keep this slice's candidates >= tau_max, in order, in the list's space (free again).
    uint64_t* kept = reinterpret_cast<uint64_t*>(list);  // LIST / 2 >= POOL entries
    int cnt = 0;
    if (U > 0) {  // uniform
      const int per = (U + NT - 1) / NT;
      const int i0 = min(tid * per, U), i1 = min(i0 + per, U);
      int n = 0;
      for (int i = i0; i < i1; ++i) n += ckey_key(pool[i]) >= tau_max ? 1 : 0;
      int at = Block<NT>::excl_scan_int(n, sh.sc.red_i, cnt);
      for (int i = i0; i < i1; ++i) {
        const uint64_t e = pool[i];
        if (ckey_key(e) >= tau_max) kept[at++] = e;
      }
    }
    if (tid < C) dsmem_st32(dsmem_addr(&sh.sx_cnt[crank], tid), static_cast<uint32_t>(cnt));
    cta_sync<NT>();
    cluster_sync_all();  // (2) every slice's count of kept candidates is published
    int total = 0, off = 0;
    for (int c = 0; c < C; ++c) {
      off += c < crank ? sh.sx_cnt[c] : 0;
      total += sh.sx_cnt[c];
    }
    const bool complete = worst == 0 && total <= POOL;  // the same in every CTA of the cluster
    if (complete) {  // each slice stores its kept candidates at its place in the first CTA's pool
      const uint32_t base = dsmem_addr(pool + off, 0);
      for (int i = tid; i < cnt; i += NT) dsmem_st64(base + 8u * static_cast<uint32_t>(i), kept[i]);
    }
    cta_sync<NT>();
    cluster_sync_all();  // (3) the first CTA's pool is complete; no other CTA's memory is used after this
    if (crank != 0) return;

    // ---- the first CTA finishes the row ----
    float m_all = -INFINITY, Z_all = 0.f;
    for (int c = 0; c < C; ++c) stat_merge(m_all, Z_all, sh.sx_m[c], sh.sx_Z[c], rc.c);  // slice order
    if (worst == -2) {
      if (tid == 0) {
        p.tokens[row] = -1;
        p.row_status[row] = kRowTimeout;
        if (p.lengths) p.lengths[row] = 0;
      }
      return;
    }
    if (!(m_all > -INFINITY && m_all < INFINITY) || !(Z_all == Z_all)) {
      if (tid == 0) write_bad_row(p, row, rc.capture);
      return;
    }
    if (tid == 0) {
      sh.row_m = m_all;
      sh.row_Z = Z_all;
    }
    const BinsPlan bins = bins_plan(rc, tau_max, m_all, DT == 0);
    if (complete && bins.dense) {  // uniform: the presence bits of the merged candidates
      for (int i = tid; i < bins.nw; i += NT) bitmap[i] = 0;
      cta_sync<NT>();
      for (int i = tid; i < total; i += NT) {
        const int d = bins.m16 - static_cast<int>(ckey_key(pool[i]) >> 16);
        atomicOr(&bitmap[d >> 5], 1u << (d & 31));
      }
    }
    cta_sync<NT>();  // also publishes sh.row_m / sh.row_Z
    if (DT == 0 && complete && bins.ok) {
      const int Q = (total + NW - 1) / NW;
      if (finish_bins<NT, DYN - POOL * 8, BITW>(p, rc, pool, Q, total, sh, bins, m_all, Z_all, ring + POOL * 8, bitmap))
        return;
    }
    finish_row<DT, NT, AREA>(p, rc, pool, total, complete, sh, tau_max);
    return;
  }

  // NaN (poisons the sum), +inf (becomes the maximum) or no finite logit at all.
  if (!(m > -INFINITY && m < INFINITY) || !(Z == Z)) {
    if (tid == 0) write_bad_row(p, row, rc.capture);
    return;
  }

  const BinsPlan bins = bins_plan(rc, st.tau, m, DT == 0);

  // ---- gather the candidates into the pool in ascending id order: the head scalars, the marked
  // vectors (read again), the tail scalars ----
  const int marked = build_list<NT, SB, LIST>(st, bitmap, list, bins, sh);
  bool complete = st.bits_ok && marked <= LIST;
  int U = 0;
  if (complete) {  // uniform
    const int per = (marked + NT - 1) / NT;
    if (DT == 1)  // float rows are sorted by their full keys: any pool order does
      U = gather_pool_unordered<DT, NT, 8, POOL>(st, list, marked, pool, sh);
    else
      U = per <= 2 ? gather_pool<DT, NT, 2, POOL>(st, list, marked, per, pool, sh, bins, bitmap)
                   : gather_pool<DT, NT, 8, POOL>(st, list, marked, per, pool, sh, bins, bitmap);
    complete = U >= 0;
  }
  cta_sync<NT>();  // the pool (and the presence bitmap) are complete
  if (DT == 0 && complete && bins.ok) {
    const int Q = (U + NW - 1) / NW;  // each warp takes Q consecutive candidates
    if (finish_bins<NT, DYN - POOL * 8, BITW>(p, rc, pool, Q, U, sh, bins, m, Z, ring + POOL * 8, bitmap)) return;
  }
  finish_row<DT, NT, AREA>(p, rc, pool, U, complete, sh, st.tau);
}

}  // namespace sfc
