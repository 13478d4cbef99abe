// Element-wise kernels: the SwiGLU backward of kept rows, and the FP8 row and column quantisers.
//
// SwiGLU backward of the rows whose gate/up pre-activations the forward kept (MoEBlaze,
// Methodology item 2: the checkpointing choice, here made per row range instead of all-or-nothing).
//
// For kept rows the backward needs no recompute GEMM: with a, b the kept pre-activations (bf16),
// dh' = dY W_d (from the BwdDh GEMM) and g the row's gate,
//   h = silu(a) b,  dg += dh'.h,  dh = g dh',  dA = dh b silu'(a),  dB = dh silu(a),  Hg = g h,
// where silu'(a) = s (1 + a (1 - s)), s = 1/(1 + e^-a) -- the element-wise tail of the recompute
// GEMM's epilogue.  A warp owns a row and walks it in 16-byte vectors (coalesced), sums dh'.h in
// fp32 and leaves it in the row's first gate partial (the others zero), the layout the gate
// reduction expects.  The kept a and b come from the caller's `saved` buffer (fused layer calls) or
// from the workspace buffers that become dB and Hg (granular calls); in the second case dB and Hg
// overwrite them in place, each element read before it is written, by the same thread.
#include <algorithm>

#include <cuda_fp8.h>

#include "common.cuh"
#include "e4m3.cuh"

namespace moe {
namespace {

constexpr int kRowsPerBlock = 8;   // one warp per row

__global__ void __launch_bounds__(32 * kRowsPerBlock) swiglu_bwd_kept_kernel(
    const uint16_t* __restrict__ dh, const float* __restrict__ gate_of_prow, uint16_t* __restrict__ dA,
    const uint16_t* a_in, const uint16_t* b_in, uint16_t* dB, uint16_t* Hg, float* __restrict__ dg_part,
    const Tables* __restrict__ tb, int keep, int f, int ndg) {
  const int lane = threadIdx.x & 31;
  const int rows = min(keep, tb->total_rows);
  const int nvec = f / 8;
  for (int r = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5); r < rows; r += gridDim.x * kRowsPerBlock) {
    const float g = gate_of_prow[r];
    const size_t base = (size_t)r * f;
    float dg = 0.f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 va = reinterpret_cast<const uint4*>(a_in + base)[v];
      const uint4 vb = reinterpret_cast<const uint4*>(b_in + base)[v];
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
          const float sg = sigmoid_fast(a);
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
      reinterpret_cast<uint4*>(dB + base)[v] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      reinterpret_cast<uint4*>(Hg + base)[v] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, off);
    for (int q = lane; q < ndg; q += 32) dg_part[(size_t)r * ndg + q] = q == 0 ? dg : 0.f;
  }
}

// FP8 rows (the quantisation step of the e4m3 expert GEMMs): per row, amax over the row, scale =
// amax / 448 in fp32 (1 for an all-zero row), codes = e4m3(v / scale) rounded to nearest even and
// saturated.  A block owns a row at a time and keeps it in registers (NV 16-byte vectors of eight
// values per thread) between the amax and the encode, so each value crosses HBM once in each
// direction; the block's next row is loaded while the current one is reduced and encoded, so two
// rows a block are in flight (one row a block left the kernel at about half the copy bandwidth).
// With the dispatch tables given, rows past the padded expert rows of this step (tb->total_rows)
// are skipped.
constexpr int kQuantV = 8;   // the most vectors a thread holds (512 threads: 32768 values a row)

template <int NV>
__device__ __forceinline__ void load_row(const uint16_t* __restrict__ src, int cols1, const uint16_t* __restrict__ src2,
                                         int cols2, int64_t r, int nvec1, int nvec, int nthreads, uint4 (&v)[NV]) {
  const uint4* row = reinterpret_cast<const uint4*>(src + r * cols1);
  const uint4* row2 = reinterpret_cast<const uint4*>(src2 + r * cols2);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int q = threadIdx.x + i * nthreads;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (q < nvec) v[i] = q < nvec1 ? row[q] : row2[q - nvec1];
  }
}

template <int kThreads, int NV>
__global__ void __launch_bounds__(kThreads) quantize_rows_e4m3_kernel(const uint16_t* __restrict__ src, int cols1,
                                                                      const uint16_t* __restrict__ src2, int cols2,
                                                                      int64_t rows, uint8_t* __restrict__ codes,
                                                                      float* __restrict__ scales,
                                                                      const Tables* __restrict__ tb) {
  constexpr int kWarps = kThreads / 32;
  __shared__ float part[2][kWarps];   // per-warp maxima, double-buffered across rows
  if (tb != nullptr) rows = min(rows, (int64_t)tb->total_rows);
  // a row is src's row (cols1 values) followed by src2's (cols2 values, often none)
  const int nvec1 = cols1 / 8, nvec = (cols1 + cols2) / 8;
  const int cols = cols1 + cols2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int buf = 0;
  uint4 v[NV], nx[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) nx[i] = make_uint4(0u, 0u, 0u, 0u);
  if ((int64_t)blockIdx.x < rows) load_row<NV>(src, cols1, src2, cols2, blockIdx.x, nvec1, nvec, kThreads, v);
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, buf ^= 1) {
    const int64_t rn = r + gridDim.x;
    if (rn < rows) load_row<NV>(src, cols1, src2, cols2, rn, nvec1, nvec, kThreads, nx);   // the next row, early
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) amax = fmaxf(amax, amax8_bf16(v[i]));   // zero vectors past the row
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (kWarps > 1) {
      if (lane == 0) part[buf][warp] = amax;
      __syncthreads();   // also orders the previous row's reads of part[buf ^ 1] before its next writes
#pragma unroll
      for (int w = 0; w < kWarps; ++w) amax = fmaxf(amax, part[buf][w]);
    }
    const float scale = e4m3_row_scale(amax);
    if (threadIdx.x == 0) scales[r] = scale;
    uint2* out = reinterpret_cast<uint2*>(codes + r * cols);
    if (e4m3_recip_ok(scale)) {   // the same branch for the whole block
      const float y = __frcp_rn(scale);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int q = threadIdx.x + i * kThreads;
        if (q < nvec) out[q] = encode8_e4m3<true>(v[i], scale, y);
      }
    } else {
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int q = threadIdx.x + i * kThreads;
        if (q < nvec) out[q] = encode8_e4m3<false>(v[i], scale, 0.f);
      }
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = nx[i];
  }
}

template <int kThreads, int NV>
void launch_quantize_nv(const uint16_t* src, int cols1, const uint16_t* src2, int cols2, int64_t rows, uint8_t* codes,
                        float* scales, const Tables* tabs, cudaStream_t s) {
  const int per_sm = std::min(32, 2048 / kThreads);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(rows, (int64_t)num_sms() * per_sm));
  quantize_rows_e4m3_kernel<kThreads, NV><<<(int)blocks, kThreads, 0, s>>>(src, cols1, src2, cols2, rows, codes,
                                                                          scales, tabs);
}

// vectors a thread holds: the row's vectors over the block's threads, rounded up to 1, 2, 4 or 8
template <int kThreads>
void launch_quantize(const uint16_t* src, int cols1, const uint16_t* src2, int cols2, int64_t rows, uint8_t* codes,
                     float* scales, const Tables* tabs, cudaStream_t s) {
  const int nv = ((cols1 + cols2) / 8 + kThreads - 1) / kThreads;
  if (nv <= 1) launch_quantize_nv<kThreads, 1>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else if (nv <= 2) launch_quantize_nv<kThreads, 2>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else if (nv <= 4) launch_quantize_nv<kThreads, 4>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else launch_quantize_nv<kThreads, kQuantV>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
}

// ---- columns: per-column e4m3 codes written transposed (the K-major operand whose rows are the
// source's columns), for the backward's weights: W_d's columns (one scale per d_ff channel) and
// column i of W_gate and W_up together (one scale per d_model channel).  The source of expert g is
// [top[g] (rows_top rows); bottom[g] (rows_bot rows)], [rows, cols] bf16; codes[g] is [cols, rows].
// Three passes: column maxima (atomicMax on the bit patterns of non-negative floats, which order
// like the values, so the result does not depend on the order of the blocks); the encode, 64 rows
// x 32 columns per block, transposed through shared memory; the scales from the maxima.

constexpr int kColRows = 256;   // rows per block of the column-maximum pass

__device__ __forceinline__ float col_src(const uint16_t* top, const uint16_t* bot, int g, int rt, int rb, int cols,
                                         int r, int c) {
  const uint16_t u = r < rt ? top[((size_t)g * rt + r) * cols + c] : bot[((size_t)g * rb + (r - rt)) * cols + c];
  return __uint_as_float((uint32_t)u << 16);
}

__global__ void col_amax_kernel(const uint16_t* __restrict__ top, const uint16_t* __restrict__ bot, int rt, int rb,
                                int cols, uint32_t* __restrict__ amax_bits) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.z;
  if (c >= cols) return;
  const int r0 = blockIdx.y * kColRows, r1 = min(rt + rb, r0 + kColRows);
  float m = 0.f;
  for (int r = r0; r < r1; ++r) m = fmaxf(m, fabsf(col_src(top, bot, g, rt, rb, cols, r, c)));
  atomicMax(&amax_bits[(size_t)g * cols + c], __float_as_uint(m));
}

// 32 x 8 threads; a block encodes rows [r0, r0 + 64) of columns [c0, c0 + 32) of expert g
__global__ void col_encode_kernel(const uint16_t* __restrict__ top, const uint16_t* __restrict__ bot, int rt, int rb,
                                  int cols, const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes) {
  __shared__ uint8_t tile[32][64 + 16];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int rows = rt + rb;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 64, g = blockIdx.z;
  const int c = c0 + tx;
  float scale = 1.f, y = 1.f;
  if (c < cols) {
    const float amax = __uint_as_float(amax_bits[(size_t)g * cols + c]);
    scale = e4m3_row_scale(amax);
    y = __frcp_rn(scale);
  }
  const bool recip = e4m3_recip_ok(scale);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int rr = 2 * ty + 16 * k;   // this thread's row pair within the tile
    const int r = r0 + rr;
    float v0 = 0.f, v1 = 0.f;
    if (c < cols && r < rows) v0 = col_src(top, bot, g, rt, rb, cols, r, c);
    if (c < cols && r + 1 < rows) v1 = col_src(top, bot, g, rt, rb, cols, r + 1, c);
    const float2 f2 = recip ? make_float2(div_by_scale(v0, scale, y), div_by_scale(v1, scale, y))
                            : make_float2(__fdiv_rn(v0, scale), __fdiv_rn(v1, scale));
    const uint32_t cc = (uint32_t)__nv_cvt_float2_to_fp8x2(f2, __NV_SATFINITE, __NV_E4M3);
    tile[tx][rr] = (uint8_t)(cc & 0xFFu);
    tile[tx][rr + 1] = (uint8_t)(cc >> 8);
  }
  __syncthreads();
  // column c0 + j gets codes of rows r0 .. r0 + 63: eight bytes per thread, 256 threads = 32 x 64
  const int j = threadIdx.x >> 3, part = threadIdx.x & 7;
  const int cc = c0 + j, rr = r0 + part * 8;
  if (cc >= cols || rr >= rows) return;
  uint8_t* dst = codes + ((size_t)g * cols + cc) * rows + rr;
  if (rr + 8 <= rows) {
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      w0 |= (uint32_t)tile[j][part * 8 + b] << (8 * b);
      w1 |= (uint32_t)tile[j][part * 8 + 4 + b] << (8 * b);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);   // rows is a multiple of 16: 8-byte aligned
  } else {
    for (int b = 0; rr + b < rows; ++b) dst[b] = tile[j][part * 8 + b];
  }
}

__global__ void col_scales_kernel(const uint32_t* __restrict__ amax_bits, float* __restrict__ scales, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float amax = __uint_as_float(amax_bits[i]);
    scales[i] = e4m3_row_scale(amax);
  }
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const uint16_t* src, int64_t rows, int cols, uint8_t* codes, float* scales,
                                      cudaStream_t s, const Tables* tabs) {
  return launch_quantize_rows2_e4m3(src, cols, nullptr, 0, rows, codes, scales, s, tabs);
}

cudaError_t launch_quantize_rows2_e4m3(const uint16_t* src, int cols1, const uint16_t* src2, int cols2, int64_t rows,
                                       uint8_t* codes, float* scales, cudaStream_t s, const Tables* tabs) {
  if (rows <= 0) return cudaSuccess;
  // threads per row: about four vectors each, between one warp and 512 threads (eight vectors
  // each at the widest row, 32768 values)
  const int nvec = (cols1 + cols2) / 8;
  if (nvec > kQuantV * 512 || cols1 % 8 != 0 || cols2 % 8 != 0) return cudaErrorInvalidValue;
  prof_mark(kKQuantE4m3, s, true);
  if (nvec <= 4 * 32) launch_quantize<32>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else if (nvec <= 4 * 64) launch_quantize<64>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else if (nvec <= 4 * 128) launch_quantize<128>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else if (nvec <= kQuantV * 256) launch_quantize<256>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  else launch_quantize<512>(src, cols1, src2, cols2, rows, codes, scales, tabs, s);
  prof_mark(kKQuantE4m3, s, false);
  return cudaGetLastError();
}

cudaError_t launch_quantize_cols_e4m3(const uint16_t* top, const uint16_t* bottom, int64_t G, int rows_top,
                                      int rows_bot, int cols, uint8_t* codes, float* scales, cudaStream_t s) {
  if (G <= 0) return cudaSuccess;
  const int rows = rows_top + rows_bot;
  // the maxima are collected in `scales` (as bit patterns), then turned into scales in place
  uint32_t* amax = reinterpret_cast<uint32_t*>(scales);
  cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)G * cols * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  prof_mark(kKQuantCols, s, true);
  col_amax_kernel<<<dim3((cols + 255) / 256, (rows + kColRows - 1) / kColRows, (unsigned)G), 256, 0, s>>>(
      top, bottom, rows_top, rows_bot, cols, amax);
  col_encode_kernel<<<dim3((cols + 31) / 32, (rows + 63) / 64, (unsigned)G), 256, 0, s>>>(top, bottom, rows_top,
                                                                                         rows_bot, cols, amax, codes);
  const int64_t n = G * (int64_t)cols;
  col_scales_kernel<<<(int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8)), 256, 0, s>>>(
      amax, scales, n);
  prof_mark(kKQuantCols, s, false);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd_kept(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s) {
  const int keep = (int)std::min<int64_t>(c.keep, L.rows);
  if (keep <= 0) return cudaSuccess;
  const int blocks = std::max(1, std::min((keep + kRowsPerBlock - 1) / kRowsPerBlock, num_sms() * 8));
  prof_mark(kKSwigluKept, s, true);
  const uint16_t* a_in = a.a_kept != nullptr ? a.a_kept : a.dB;
  const uint16_t* b_in = a.b_kept != nullptr ? a.b_kept : a.Hg;
  swiglu_bwd_kept_kernel<<<blocks, 32 * kRowsPerBlock, 0, s>>>(a.dh, a.gate_of_prow, a.dA, a_in, b_in, a.dB,
                                                              a.Hg, a.dg_part, a.tabs, keep, c.f, L.ndg);
  prof_mark(kKSwigluKept, s, false);
  return cudaGetLastError();
}

}  // namespace moe
