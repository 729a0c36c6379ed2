// Training-side replay: the sampled token's log-probability under a policy's logits renormalised
// over a captured support ("vLLM Sampling Mask（Distribution Replay）深入解析", section RL 训练侧使用:
// every token outside the support is masked to -inf before the log-softmax, which is read at the
// sampled token).
//
// One CTA of 256 threads per row. The support's ids are read coalesced, the logits they name are
// gathered (up to eight loads in flight per thread, so a 2048-entry support is one round trip), and
// an online (max, sum of 2^((x - m) c)) state per thread is merged by warp butterflies and then
// across the warps in a fixed order, so results are deterministic. A second gather writes the
// support's log-probabilities when they are asked for.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sfc.h"
#include "sfc_device.cuh"

namespace sfc {
namespace {

struct ReplayParams {
  const void* logits;
  int64_t row_stride, V;
  int32_t B, W;
  const float* temperature;
  const int32_t* support_ids;
  const int32_t* lengths;
  const int32_t* tokens;
  float* token_logprob;
  float* support_logprobs;
  int32_t* row_status;
};

constexpr int kReplayThreads = 256;
constexpr int kReplayUnroll = 8;
constexpr float kLog2eF = 1.4426950408889634f;

template <int DT>
__device__ __forceinline__ float replay_logit(const unsigned char* row, int32_t id) {
  return Elem<DT>::load1(row, id);
}

template <int DT>
__global__ void __launch_bounds__(kReplayThreads) replay_kernel(const __grid_constant__ ReplayParams p) {
  constexpr int NW = kReplayThreads / 32;
  __shared__ float red_m[NW], red_s[NW], red_x[NW];
  __shared__ int red_f[NW];
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  const int r = blockIdx.x;
  const float T = p.temperature[r];
  const int n = p.lengths[r];
  const int32_t tok = p.tokens[r];
  auto finish = [&](int status, float lp) {
    if (tid == 0) {
      p.row_status[r] = status;
      p.token_logprob[r] = lp;
    }
  };
  if (!(T > 0.f && T < INFINITY) || n < 1) return finish(SFC_ROW_BADPARAM, __int_as_float(0x7fc00000));
  if (n > p.W) return finish(SFC_ROW_OVERFLOW, __int_as_float(0x7fc00000));
  const unsigned char* row = static_cast<const unsigned char*>(p.logits) + static_cast<int64_t>(r) * p.row_stride * Elem<DT>::kBytes;
  const int32_t* ids = p.support_ids + static_cast<int64_t>(r) * p.W;
  const float c = kLog2eF / T;
  // Pass 1: online maximum and mass per thread, the token's logit, checks.
  float m = -INFINITY, s = 0.f, x_tok = 0.f;
  int flags = 0;  // bit 0: a bad id or logit; bit 1: the token was found
  for (int j0 = 0; j0 < n; j0 += kReplayThreads * kReplayUnroll) {  // uniform
    int32_t id[kReplayUnroll];
    float x[kReplayUnroll];
#pragma unroll
    for (int u = 0; u < kReplayUnroll; ++u) {
      const int j = j0 + kReplayThreads * u + tid;
      id[u] = j < n ? ids[j] : -1;
    }
#pragma unroll
    for (int u = 0; u < kReplayUnroll; ++u) {
      const bool in = id[u] >= 0 && static_cast<int64_t>(id[u]) < p.V;
      if (j0 + kReplayThreads * u + tid < n && !in) flags |= 1;
      const float v = replay_logit<DT>(row, in ? id[u] : 0);  // always a valid address
      x[u] = in ? v : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kReplayUnroll; ++u) {
      if (!(x[u] < INFINITY)) flags |= 1;  // NaN or +inf
      if (id[u] == tok && tok >= 0) {
        flags |= 2;
        x_tok = x[u];
      }
      if (x[u] > m) {
        s = (m > -INFINITY) ? s * ex2_approx((m - x[u]) * c) : 0.f;
        m = x[u];
      }
      s += ex2_approx((x[u] - m) * c);  // -inf gives 0
    }
  }
  // Merge: warp butterflies, then the warps in order.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(kFull, m, o), s2 = __shfl_xor_sync(kFull, s, o);
    stat_merge(m, s, m2, s2, c);
  }
  const int any_bad = __any_sync(kFull, flags & 1);
  const unsigned hit = __ballot_sync(kFull, flags & 2);
  if (hit) x_tok = __shfl_sync(kFull, x_tok, __ffs(static_cast<int>(hit)) - 1);  // warp-uniform
  if (lane == 0) {
    red_m[wp] = m;
    red_s[wp] = s;
    red_f[wp] = any_bad | (hit ? 2 : 0);
    red_x[wp] = x_tok;
  }
  __syncthreads();
  m = red_m[0];
  s = red_s[0];
  int fl = red_f[0];
  if (fl & 2) x_tok = red_x[0];
  for (int v = 1; v < NW; ++v) {
    stat_merge(m, s, red_m[v], red_s[v], c);
    if (!(fl & 2) && (red_f[v] & 2)) x_tok = red_x[v];
    fl |= red_f[v];
  }
  if ((fl & 1) || !(m > -INFINITY)) return finish(SFC_ROW_BADPARAM, __int_as_float(0x7fc00000));
  const float lnZ = logf(s);  // ln sum exp((x - m) / T)
  if (p.support_logprobs) {  // pass 2: every member's log-probability
    float* out = p.support_logprobs + static_cast<int64_t>(r) * p.W;
    for (int j = tid; j < n; j += kReplayThreads) out[j] = (replay_logit<DT>(row, ids[j]) - m) / T - lnZ;
  }
  if (fl & 2) return finish(SFC_ROW_OK, (x_tok - m) / T - lnZ);
  finish(SFC_ROW_OUTSIDE, -INFINITY);
}

}  // namespace
}  // namespace sfc

extern "C" int sfc_replay_logprob(const void* logits, int dtype, int64_t B, int64_t V, int64_t row_stride,
                                  const float* temperature, const int32_t* support_ids, const int32_t* lengths,
                                  int32_t packed_width, const int32_t* tokens, float* token_logprob,
                                  float* support_logprobs, int32_t* row_status, void* stream) {
  if (!logits || !temperature || !support_ids || !lengths || !tokens || !token_logprob || !row_status)
    return SFC_EINVAL;
  if (dtype != SFC_BF16 && dtype != SFC_F32) return SFC_EINVAL;
  if (B < 1 || B > INT32_MAX || V < 1 || V > INT32_MAX || row_stride < V) return SFC_EINVAL;
  if (packed_width < 1 || packed_width > SFC_MAX_PACKED_WIDTH) return SFC_EINVAL;
  const int elt = dtype == SFC_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % elt) return SFC_EINVAL;
  sfc::ReplayParams p;
  p.logits = logits;
  p.row_stride = row_stride;
  p.V = V;
  p.B = static_cast<int32_t>(B);
  p.W = packed_width;
  p.temperature = temperature;
  p.support_ids = support_ids;
  p.lengths = lengths;
  p.tokens = tokens;
  p.token_logprob = token_logprob;
  p.support_logprobs = support_logprobs;
  p.row_status = row_status;
  const unsigned grid = static_cast<unsigned>(B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SFC_BF16)
    sfc::replay_kernel<0><<<grid, sfc::kReplayThreads, 0, st>>>(p);
  else
    sfc::replay_kernel<1><<<grid, sfc::kReplayThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SFC_ECUDA;
  return SFC_OK;
}
