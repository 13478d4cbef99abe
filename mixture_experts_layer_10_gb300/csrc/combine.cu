// Combine (reverse dispatch) by token owner, and the gate-gradient reduction of the backward.
//
// Each block owns 32 tokens x 256 columns; a thread owns 4 tokens x 8 columns and reads each of
// its tokens' expert rows with 16-byte loads, in fixed slot order, accumulating in fp32 and
// rounding once to bf16.  No atomics: the result is bitwise deterministic.  Sources: MoEBlaze
// (Methodology item 2: scatter/gather around the expert FFN) and the DisagMoE summary (section 2.2:
// combine after the experts).  The input-gradient combine of the backward is the same kernel with
// unit weights and one more source row per token: the router's dlogits W_r^T, computed on the
// tensor cores beforehand (RouterDx in gemm.cu).
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kTokTile = 32;
constexpr int kColTile = 256;

__device__ __forceinline__ void add_vec8(float (&acc)[8], const uint4& v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    acc[2 * m] = fmaf(w, bf16_lo(u[m]), acc[2 * m]);
    acc[2 * m + 1] = fmaf(w, bf16_hi(u[m]), acc[2 * m + 1]);
  }
}

__device__ __forceinline__ void add_row8(float (&acc)[8], const uint16_t* row, float w) {
  add_vec8(acc, *reinterpret_cast<const uint4*>(row), w);
}

__device__ __forceinline__ void store_row8(uint16_t* row, const float (&acc)[8]) {
  uint4 v;
  v.x = pack_bf16(acc[0], acc[1]);
  v.y = pack_bf16(acc[2], acc[3]);
  v.z = pack_bf16(acc[4], acc[5]);
  v.w = pack_bf16(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(row) = v;
}

// y[t] = extra[t] + sum_j gates[t,j] * rows[prow(t,j)] + sum_s rows[P_{E+s} + t], with extra
// (a [T, d] bf16 row per token) and gates (weight 1 when null) optional.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const float* __restrict__ gates,
                                                      const uint16_t* __restrict__ extra,
                                                      uint16_t* __restrict__ out,
                                                      const Tables* __restrict__ tb,
                                                      const int32_t* __restrict__ prow_of_slot,
                                                      int T, int d, int k, int E, int S) {
  const int tx = threadIdx.x & 31;          // 8-column group
  const int ty = threadIdx.x >> 5;          // 4-token group
  const int t0 = blockIdx.x * kTokTile;
  const int col = blockIdx.y * kColTile + tx * 8;
  if (col >= d) return;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) break;
    float acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = 0.f;
    if (extra != nullptr) add_row8(acc, extra + (size_t)t * d + col, 1.f);
    // slots in groups of four: the four rows are loaded before any is added (more bytes in
    // flight per thread), then added in slot order
    for (int j0 = 0; j0 < k; j0 += 4) {
      uint4 v[4];
      float w[4];
      bool has[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        v[u] = make_uint4(0, 0, 0, 0);
        w[u] = 0.f;
        has[u] = false;
        if (j < k) {
          const size_t slot = (size_t)t * k + j;
          const int p = prow_of_slot[slot];
          if (p >= 0) {
            v[u] = *reinterpret_cast<const uint4*>(rows + (size_t)p * d + col);
            w[u] = gates != nullptr ? gates[slot] : 1.f;
            has[u] = true;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (has[u]) add_vec8(acc, v[u], w[u]);
    }
    for (int s = 0; s < S; ++s) {
      if (t >= tb->kept[E + s]) continue;
      add_row8(acc, rows + ((size_t)tb->poff[E + s] + t) * d + col, 1.f);
    }
    store_row8(out + (size_t)t * d + col, acc);
  }
}

// dgates[t,j] = sum over the d_ff tiles of the per-row partials dy.o written by the backward
// GEMM's epilogue (0 for dropped slots).  kG lanes own a slot: lane i of the group reads partials
// i, i + kG, ... of the row (coalesced, several loads in flight per lane), and a shuffle tree of
// fixed shape joins the group; the order is fixed, so the result is deterministic.
template <int kG>
__global__ void dgates_kernel(const float* __restrict__ dg_part, const int32_t* __restrict__ prow_of_slot,
                              float* __restrict__ dgates, int n, int ntf) {
  const int sub = threadIdx.x & (kG - 1);
  const int g0 = (int)((blockIdx.x * blockDim.x + threadIdx.x) / kG);
  const int ng = (int)((gridDim.x * blockDim.x) / kG);
  for (int i0 = g0 - (g0 % (32 / kG)); i0 < n; i0 += ng) {   // whole warps iterate together
    const int i = i0 + (g0 % (32 / kG));
    const int p = i < n ? prow_of_slot[i] : -1;
    float v = 0.f;
    if (p >= 0) {
#pragma unroll 4
      for (int q = sub; q < ntf; q += kG) v += dg_part[(size_t)p * ntf + q];
    }
#pragma unroll
    for (int off = kG / 2; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off, kG);
    if (sub == 0 && i < n) dgates[i] = v;
  }
}

}  // namespace

cudaError_t launch_combine(const Cfg& c, const CombineArgs& a, cudaStream_t s) {
  dim3 grid((c.T + kTokTile - 1) / kTokTile, (c.d + kColTile - 1) / kColTile);
  prof_mark(kKCombine, s, true);
  combine_kernel<<<grid, 256, 0, s>>>(a.o_perm, a.gates, nullptr, a.y, a.tabs, a.prow_of_slot, c.T, c.d, c.k,
                                      c.E, c.S);
  prof_mark(kKCombine, s, false);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Cfg& c, const CombineBwdArgs& a, cudaStream_t s) {
  dim3 grid((c.T + kTokTile - 1) / kTokTile, (c.d + kColTile - 1) / kColTile);
  prof_mark(kKCombineBwd, s, true);
  combine_kernel<<<grid, 256, 0, s>>>(a.dx_perm, nullptr, a.r, a.dx, a.tabs, a.prow_of_slot, c.T, c.d, c.k,
                                      c.E, c.S);
  prof_mark(kKCombineBwd, s, false);
  return cudaGetLastError();
}

cudaError_t launch_dgates(const Cfg& c, const Layout& L, const DgatesArgs& a, cudaStream_t s) {
  const int n = c.T * c.k;
  // lanes per slot: the largest power of two that leaves each lane about six of the row's partials
  // (memory-level parallelism), at most a warp
  int g = 1;
  while (g < 32 && 2 * g * 6 <= L.ndg) g *= 2;
  const long long threads = (long long)n * g;
  const int blocks = (int)std::max<long long>(1, std::min<long long>((threads + 255) / 256, (long long)num_sms() * 16));
  prof_mark(kKDgates, s, true);
  switch (g) {
    case 32: dgates_kernel<32><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
    case 16: dgates_kernel<16><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
    case 8: dgates_kernel<8><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
    case 4: dgates_kernel<4><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
    case 2: dgates_kernel<2><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
    default: dgates_kernel<1><<<blocks, 256, 0, s>>>(a.dg_part, a.prow_of_slot, a.dgates, n, L.ndg); break;
  }
  prof_mark(kKDgates, s, false);
  return cudaGetLastError();
}

}  // namespace moe
