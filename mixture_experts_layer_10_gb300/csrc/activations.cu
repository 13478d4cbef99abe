// SwiGLU backward of the rows whose gate/up pre-activations the forward kept (MoEBlaze,
// Methodology item 2: the checkpointing choice, here made per row range instead of all-or-nothing).
//
// For kept rows the backward needs no recompute GEMM: with a, b the kept pre-activations (bf16),
// dh' = dY W_d (from the BwdDh GEMM) and g the row's gate,
//   h = silu(a) b,  dg += dh'.h,  dh = g dh',  dA = dh b silu'(a),  dB = dh silu(a),  Hg = g h,
// where silu'(a) = s (1 + a (1 - s)), s = 1/(1 + e^-a) -- the element-wise tail of the recompute
// GEMM's epilogue.  A warp owns a row and walks it in 16-byte vectors (coalesced), sums dh'.h in
// fp32 and leaves it in the row's first gate partial (the others zero), the layout the gate
// reduction expects.  dB and Hg overwrite the kept a and b in place: each element is read before
// it is written, by the same thread.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRowsPerBlock = 8;   // one warp per row

__global__ void __launch_bounds__(32 * kRowsPerBlock) swiglu_bwd_kept_kernel(
    const uint16_t* __restrict__ dh, const float* __restrict__ gate_of_prow, uint16_t* __restrict__ dA,
    uint16_t* __restrict__ a_dB, uint16_t* __restrict__ b_Hg, float* __restrict__ dg_part,
    const Tables* __restrict__ tb, int keep, int f, int ndg) {
  const int lane = threadIdx.x & 31;
  const int rows = min(keep, tb->total_rows);
  const int nvec = f / 8;
  for (int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); r < rows; r += gridDim.x * kRowsPerBlock) {
    const float g = gate_of_prow[r];
    const size_t base = (size_t)r * f;
    float dg = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 va = reinterpret_cast<const uint4*>(a_dB + base)[v];
      const uint4 vb = reinterpret_cast<const uint4*>(b_Hg + base)[v];
      const uint4 vd = reinterpret_cast<const uint4*>(dh + base)[v];
      const uint32_t ua[4] = {va.x, va.y, va.z, va.w};
      const uint32_t ub[4] = {vb.x, vb.y, vb.z, vb.w};
      const uint32_t ud[4] = {vd.x, vd.y, vd.z, vd.w};
      uint32_t oa[4], ob[4], oh[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        float o_da[2], o_db[2], o_h[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float a = h ? bf16_hi(ua[m]) : bf16_lo(ua[m]);
          const float b = h ? bf16_hi(ub[m]) : bf16_lo(ub[m]);
          const float dhp = h ? bf16_hi(ud[m]) : bf16_lo(ud[m]);
          const float sg = 1.f / (1.f + __expf(-a));
          const float sa = a * sg;
          const float hv = sa * b;
          dg = fmaf(dhp, hv, dg);
          const float dhv = g * dhp;
          o_da[h] = dhv * b * sg * (1.f + a * (1.f - sg));
          o_db[h] = dhv * sa;
          o_h[h] = g * hv;
        }
        oa[m] = pack_bf16(o_da[0], o_da[1]);
        ob[m] = pack_bf16(o_db[0], o_db[1]);
        oh[m] = pack_bf16(o_h[0], o_h[1]);
      }
      reinterpret_cast<uint4*>(dA + base)[v] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
      reinterpret_cast<uint4*>(a_dB + base)[v] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      reinterpret_cast<uint4*>(b_Hg + base)[v] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, off);
    for (int q = lane; q < ndg; q += 32) dg_part[(size_t)r * ndg + q] = q == 0 ? dg : 0.f;
  }
}

}  // namespace

cudaError_t launch_swiglu_bwd_kept(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s) {
  const int keep = (int)std::min<int64_t>(c.keep, L.rows);
  if (keep <= 0) return cudaSuccess;
  const int blocks = std::max(1, std::min((keep + kRowsPerBlock - 1) / kRowsPerBlock, num_sms() * 8));
  prof_mark(kKSwigluKept, s, true);
  swiglu_bwd_kept_kernel<<<blocks, 32 * kRowsPerBlock, 0, s>>>(a.dh, a.gate_of_prow, a.dA, a.dB, a.Hg,
                                                              a.dg_part, a.tabs, keep, c.f, L.ndg);
  prof_mark(kKSwigluKept, s, false);
  return cudaGetLastError();
}

}  // namespace moe
