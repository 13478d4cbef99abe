// Combine (reverse dispatch) by token owner, and the input-gradient combine of the backward.
//
// Each block owns 32 tokens x 256 columns; a thread owns 4 tokens x 8 columns and reads each of
// its tokens' expert rows with 16-byte loads, in fixed slot order, accumulating in fp32 and
// rounding once to bf16.  No atomics: the result is bitwise deterministic.  Sources: MoEBlaze
// (Methodology item 2: scatter/gather around the expert FFN) and the DisagMoE summary (section 2.2:
// combine after the experts).  The backward form adds the router's input gradient
// dlogits[t] W_r^T as a small fp32 product staged through shared memory.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kTokTile = 32;
constexpr int kColTile = 256;
constexpr int kEChunk = 32;

__device__ __forceinline__ void add_row8(float (&acc)[8], const uint16_t* row, float w) {
  const uint4 v = *reinterpret_cast<const uint4*>(row);
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    acc[2 * m] = fmaf(w, bf16_lo(u[m]), acc[2 * m]);
    acc[2 * m + 1] = fmaf(w, bf16_hi(u[m]), acc[2 * m + 1]);
  }
}

__device__ __forceinline__ void store_row8(uint16_t* row, const float (&acc)[8]) {
  uint4 v;
  v.x = pack_bf16(acc[0], acc[1]);
  v.y = pack_bf16(acc[2], acc[3]);
  v.z = pack_bf16(acc[4], acc[5]);
  v.w = pack_bf16(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(row) = v;
}

// y[t] = sum_j gates[t,j] * rows[prow(t,j)] + sum_s rows[P_{E+s} + t]   (kBwd: unit weights,
// plus dlogits[t] W_r^T).
template <bool kBwd>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const float* __restrict__ gates,
                                                      const float* __restrict__ dlogits,
                                                      const float* __restrict__ W_r,
                                                      uint16_t* __restrict__ out,
                                                      const Tables* __restrict__ tb,
                                                      const int32_t* __restrict__ prow_of_slot,
                                                      int T, int d, int k, int E, int S) {
  __shared__ float wt[kBwd ? kEChunk : 1][kColTile + 4];
  __shared__ float dl[kBwd ? kTokTile : 1][kEChunk + 1];
  const int tx = threadIdx.x & 31;          // 8-column group
  const int ty = threadIdx.x >> 5;          // 4-token group
  const int t0 = blockIdx.x * kTokTile;
  const int c0 = blockIdx.y * kColTile;
  const int col = c0 + tx * 8;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[i][m] = 0.f;

  if (kBwd && dlogits != nullptr) {
    for (int e0 = 0; e0 < E; e0 += kEChunk) {
      const int ne = min(kEChunk, E - e0);   // experts in this chunk; loads run along W_r's rows
      for (int p = threadIdx.x; p < kColTile * ne; p += 256) {
        const int i = p / ne, ee = p % ne;
        wt[ee][i] = (c0 + i < d) ? W_r[(size_t)(c0 + i) * E + e0 + ee] : 0.f;
      }
      for (int p = threadIdx.x; p < kTokTile * ne; p += 256) {
        const int tt = p / ne, ee = p % ne;
        dl[tt][ee] = (t0 + tt < T) ? dlogits[(size_t)(t0 + tt) * E + e0 + ee] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int ee = 0; ee < ne; ++ee) {
        const float4 w0 = *reinterpret_cast<const float4*>(&wt[ee][tx * 8]);
        const float4 w1 = *reinterpret_cast<const float4*>(&wt[ee][tx * 8 + 4]);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float g = dl[ty * 4 + i][ee];
#pragma unroll
          for (int m = 0; m < 8; ++m) acc[i][m] = fmaf(g, wv[m], acc[i][m]);
        }
      }
      __syncthreads();
    }
  }
  if (col >= d) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) break;
    for (int j = 0; j < k; ++j) {
      const size_t slot = (size_t)t * k + j;
      const int p = prow_of_slot[slot];
      if (p < 0) continue;
      add_row8(acc[i], rows + (size_t)p * d + col, kBwd ? 1.f : gates[slot]);
    }
    for (int s = 0; s < S; ++s) {
      if (t >= tb->kept[E + s]) continue;
      add_row8(acc[i], rows + ((size_t)tb->poff[E + s] + t) * d + col, 1.f);
    }
    store_row8(out + (size_t)t * d + col, acc[i]);
  }
}

// dgates[t,j] = sum over the d_ff tiles of the per-row partials dy.o written by the backward
// GEMM's epilogue (0 for dropped slots).
__global__ void dgates_kernel(const float* __restrict__ dg_part, const int32_t* __restrict__ prow_of_slot,
                              float* __restrict__ dgates, int n, int ntf) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int p = prow_of_slot[i];
    float v = 0.f;
    if (p >= 0)
      for (int q = 0; q < ntf; ++q) v += dg_part[(size_t)p * ntf + q];
    dgates[i] = v;
  }
}

}  // namespace

cudaError_t launch_combine(const Cfg& c, const CombineArgs& a, cudaStream_t s) {
  dim3 grid((c.T + kTokTile - 1) / kTokTile, (c.d + kColTile - 1) / kColTile);
  prof_mark(kKCombine, s, true);
  combine_kernel<false><<<grid, 256, 0, s>>>(a.o_perm, a.gates, nullptr, nullptr, a.y, a.tabs,
                                             a.prow_of_slot, c.T, c.d, c.k, c.E, c.S);
  prof_mark(kKCombine, s, false);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Cfg& c, const CombineBwdArgs& a, cudaStream_t s) {
  dim3 grid((c.T + kTokTile - 1) / kTokTile, (c.d + kColTile - 1) / kColTile);
  prof_mark(kKCombineBwd, s, true);
  combine_kernel<true><<<grid, 256, 0, s>>>(a.dx_perm, nullptr, a.dlogits, a.W_r, a.dx, a.tabs,
                                            a.prow_of_slot, c.T, c.d, c.k, c.E, c.S);
  prof_mark(kKCombineBwd, s, false);
  return cudaGetLastError();
}

cudaError_t launch_dgates(const Cfg& c, const Layout& L, const DgatesArgs& a, cudaStream_t s) {
  const int n = c.T * c.k;
  const int blocks = std::max(1, std::min((n + 255) / 256, num_sms() * 4));
  prof_mark(kKDgates, s, true);
  dgates_kernel<<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg);
  prof_mark(kKDgates, s, false);
  return cudaGetLastError();
}

}  // namespace moe
