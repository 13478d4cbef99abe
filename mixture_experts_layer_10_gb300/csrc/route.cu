// Router: logits = x W_r (+ b), softmax over the E routed experts, top-k by logit (ties to the
// lower expert index), gates; and its backward with the selection held fixed.
//
// This file holds the SIMT router, used where the tensor-core routers do not apply (more than 128
// experts, or more than 8 per token): the logits are an fp32 tile product (x is bf16, W_r fp32,
// E <= 256 columns); selection, softmax and the gate gradient run warp-per-token with shuffle
// reductions.  Up to 32 experts (k <= 8) route_tc.cu streams x on the tensor cores with K split
// across CTAs, and up to 128 experts gemm.cu's RouterLogits gives each 128-token tile a CTA; the
// W_r split kernels of both, the router-backward reductions and the bf16 row conversion are here
// too.  Sources: the Piper explainer ("the problem": a router sends each token to a few experts)
// and the MoEBlaze summary (Limitations: static top-k routing); the formulas are the plain
// softmax-then-top-k reading.
#include <algorithm>
#include <cfloat>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 64;   // k-chunk staged in shared memory (double-buffered)

// Tile shapes per expert bucket: BT tokens x EB experts per block; a thread owns TM tokens x TN
// experts and a 1/KS share of each k-chunk.
template <int EB> struct RouteShape;
template <> struct RouteShape<8>   { static constexpr int BT = 32, TM = 1, TN = 8, KS = 8; };
template <> struct RouteShape<16>  { static constexpr int BT = 32, TM = 2, TN = 8, KS = 8; };
template <> struct RouteShape<32>  { static constexpr int BT = 32, TM = 2, TN = 8, KS = 4; };
template <> struct RouteShape<64>  { static constexpr int BT = 64, TM = 4, TN = 4, KS = 1; };
template <> struct RouteShape<128> { static constexpr int BT = 64, TM = 4, TN = 8, KS = 1; };
template <> struct RouteShape<256> { static constexpr int BT = 32, TM = 4, TN = 8, KS = 1; };

template <int EB>
struct LogitSmem {
  using S = RouteShape<EB>;
  float xs[2][kKC][S::BT + 4];  // x chunk, k-major, double-buffered
  float ws[2][kKC][EB];         // W_r chunk, double-buffered
  float red[S::KS > 1 ? S::KS : 1][S::BT][EB + 1];   // k-split partials, then the logits tile
};

// One k-chunk of x (BT rows x 64 bf16, 8 16-byte pieces per row) and of W_r (64 rows x EB),
// held in registers between its global loads and its shared-memory stores.
template <int EB>
struct ChunkRegs {
  using S = RouteShape<EB>;
  static constexpr int NX = (S::BT * kKC / 8 + kThreads - 1) / kThreads;
  static constexpr int NW = (kKC * EB / 4 + kThreads - 1) / kThreads;
  uint4 x[NX];
  float4 w[NW];

  __device__ void load(const uint16_t* __restrict__ xg, const float* __restrict__ W_r, int T, int d,
                       int E, int t0, int k0) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      const int p = tid + i * kThreads;
      const int t = p % S::BT, q = p / S::BT;
      x[i] = make_uint4(0, 0, 0, 0);
      if (p < S::BT * kKC / 8 && t0 + t < T)
        x[i] = *reinterpret_cast<const uint4*>(xg + (size_t)(t0 + t) * d + k0 + q * 8);
    }
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int p = tid + i * kThreads;
      const int kk = p / (EB / 4), e = (p % (EB / 4)) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p < kKC * EB / 4) {
        const float* row = W_r + (size_t)(k0 + kk) * E;
        if ((E & 3) == 0 && e + 3 < E) {
          v = *reinterpret_cast<const float4*>(row + e);
        } else {
          if (e < E) v.x = row[e];
          if (e + 1 < E) v.y = row[e + 1];
          if (e + 2 < E) v.z = row[e + 2];
          if (e + 3 < E) v.w = row[e + 3];
        }
      }
      w[i] = v;
    }
  }

  __device__ void store(LogitSmem<EB>& sm, int buf) const {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      const int p = tid + i * kThreads;
      if (p >= S::BT * kKC / 8) break;
      const int t = p % S::BT, q = p / S::BT;
      const uint32_t u[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        sm.xs[buf][q * 8 + 2 * m][t] = bf16_lo(u[m]);
        sm.xs[buf][q * 8 + 2 * m + 1][t] = bf16_hi(u[m]);
      }
    }
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const int p = tid + i * kThreads;
      if (p >= kKC * EB / 4) break;
      const int kk = p / (EB / 4), e = (p % (EB / 4)) * 4;
      *reinterpret_cast<float4*>(&sm.ws[buf][kk][e]) = w[i];
    }
  }
};

// logits tile [BT x EB] of tokens t0.. into sm.red[0] (bias added, experts >= E left at 0).
// The next chunk's global loads are issued before the current chunk's products, and the chunks
// alternate between two shared-memory buffers (one barrier per chunk).
template <int EB>
__device__ void logits_tile(LogitSmem<EB>& sm, const uint16_t* __restrict__ x,
                            const float* __restrict__ W_r, const float* __restrict__ b_r, int T,
                            int d, int E, int t0) {
  using S = RouteShape<EB>;
  constexpr int TX = S::BT / S::TM, TY = EB / S::TN;
  static_assert(TX * TY * S::KS == kThreads, "thread tiling");
  const int tid = threadIdx.x;
  const int ks = tid / (TX * TY);
  const int ty = (tid / TX) % TY;
  const int tx = tid % TX;
  float acc[S::TM][S::TN];
#pragma unroll
  for (int i = 0; i < S::TM; ++i)
#pragma unroll
    for (int j = 0; j < S::TN; ++j) acc[i][j] = 0.f;

  ChunkRegs<EB> regs;
  regs.load(x, W_r, T, d, E, t0, 0);
  regs.store(sm, 0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < d; k0 += kKC) {
    const bool more = k0 + kKC < d;
    if (more) regs.load(x, W_r, T, d, E, t0, k0 + kKC);
    // two-level sum: each 64-wide chunk is summed on its own, then added to the running total,
    // which keeps the fp32 rounding of d-long dot products (the gates need 1e-5) several times smaller
    float part[S::TM][S::TN];
#pragma unroll
    for (int i = 0; i < S::TM; ++i)
#pragma unroll
      for (int j = 0; j < S::TN; ++j) part[i][j] = 0.f;
#pragma unroll 4
    for (int kk = ks; kk < kKC; kk += S::KS) {
      float xv[S::TM], wv[S::TN];
#pragma unroll
      for (int i = 0; i < S::TM; ++i) xv[i] = sm.xs[buf][kk][tx * S::TM + i];
#pragma unroll
      for (int j = 0; j < S::TN; ++j) wv[j] = sm.ws[buf][kk][ty * S::TN + j];
#pragma unroll
      for (int i = 0; i < S::TM; ++i)
#pragma unroll
        for (int j = 0; j < S::TN; ++j) part[i][j] = fmaf(xv[i], wv[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < S::TM; ++i)
#pragma unroll
      for (int j = 0; j < S::TN; ++j) acc[i][j] += part[i][j];
    if (more) regs.store(sm, buf ^ 1);   // that buffer was last read before the previous barrier
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < S::TM; ++i)
#pragma unroll
    for (int j = 0; j < S::TN; ++j) sm.red[ks][tx * S::TM + i][ty * S::TN + j] = acc[i][j];
  __syncthreads();
  // fixed-order k-split reduction plus bias
  for (int p = tid; p < S::BT * EB; p += kThreads) {
    const int t = p / EB, e = p % EB;
    float v = sm.red[0][t][e];
#pragma unroll
    for (int s = 1; s < S::KS; ++s) v += sm.red[s][t][e];
    if (b_r != nullptr && e < E) v += b_r[e];
    sm.red[0][t][e] = v;
  }
  __syncthreads();
}

constexpr int vals_per_lane(int EB) { return EB >= 32 ? EB / 32 : 1; }

// Warp-wide (value, index) argmax: larger value wins, equal values go to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

template <int EB>
__global__ void __launch_bounds__(kThreads) route_fwd_kernel(RouteArgs a, int T, int d, int E,
                                                             int k, int renorm) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  LogitSmem<EB>& sm = *reinterpret_cast<LogitSmem<EB>*>(smem_raw);
  using S = RouteShape<EB>;
  constexpr int NV = vals_per_lane(EB);
  const int t0 = blockIdx.x * S::BT;
  logits_tile<EB>(sm, a.x, a.W_r, a.b_r, T, d, E, t0);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int tt = warp; tt < S::BT; tt += kThreads / 32) {
    const int t = t0 + tt;
    if (t >= T) break;
    float v[NV];
    int slot[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? sm.red[0][tt][e] : -INFINITY;
      slot[i] = -1;
      if (a.logits != nullptr && e < E) a.logits[(size_t)t * E + e] = v[i];
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NV; ++i) m = fmaxf(m, v[i]);
    m = warp_max(m);
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) z += (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
    z = warp_sum(z);
    // top-k: k rounds of warp argmax over the not-yet-selected experts
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && slot[i] < 0 && (v[i] > bv || (v[i] == bv && e < bi))) {
          bv = v[i];
          bi = e;
        }
      }
      warp_argmax(bv, bi);
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (lane + 32 * i == bi) slot[i] = r;
    }
    float zsel = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (slot[i] >= 0) zsel += expf(v[i] - m);
    zsel = warp_sum(zsel);
    const float denom = renorm ? zsel : z;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (slot[i] >= 0) {
        a.idx[(size_t)t * k + slot[i]] = lane + 32 * i;
        a.gates[(size_t)t * k + slot[i]] = expf(v[i] - m) / denom;
      }
  }
}

// Router backward, part 1: per token dlogits (recomputing the softmax when not renormalised),
// and per-block db partials.
template <int EB>
__global__ void __launch_bounds__(kThreads) router_dlogits_kernel(RouterBwdArgs a, int T, int d,
                                                                  int E, int k, int renorm) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  LogitSmem<EB>& sm = *reinterpret_cast<LogitSmem<EB>*>(smem_raw);
  using S = RouteShape<EB>;
  constexpr int NV = vals_per_lane(EB);
  __shared__ float dsel[kThreads / 32][EB];
  __shared__ float dbw[kThreads / 32][EB];
  const int t0 = blockIdx.x * S::BT;
  if (!renorm) logits_tile<EB>(sm, a.x, a.W_r, a.b_r, T, d, E, t0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int e = lane; e < EB; e += 32) dbw[warp][e] = 0.f;
  __syncwarp();
  for (int tt = warp; tt < S::BT; tt += kThreads / 32) {
    const int t = t0 + tt;
    if (t >= T) break;
    // s = sum_j dg_j g_j, and dsel[e] = dg of the slot that selected e
    for (int e = lane; e < EB; e += 32) dsel[warp][e] = 0.f;
    __syncwarp();
    float s = 0.f;
    for (int j = lane; j < k; j += 32) {
      const float dg = a.dgates[(size_t)t * k + j];
      const float g = a.gates[(size_t)t * k + j];
      const int e = a.idx[(size_t)t * k + j];
      s += dg * g;
      if (e >= 0 && e < E) atomicAdd(&dsel[warp][e], renorm ? g * dg : dg);
    }
    s = warp_sum(s);
    __syncwarp();
    if (renorm) {
      // dl_{idx_j} = g_j (dg_j - s); dsel holds g_j dg_j, so subtract g_j s per selected slot
      for (int j = lane; j < k; j += 32) {
        const int e = a.idx[(size_t)t * k + j];
        if (e >= 0 && e < E) atomicAdd(&dsel[warp][e], -a.gates[(size_t)t * k + j] * s);
      }
      __syncwarp();
      for (int e = lane; e < E; e += 32) {
        const float dl = dsel[warp][e];
        a.dlogits[(size_t)t * E + e] = dl;
        dbw[warp][e] += dl;
      }
    } else {
      float v[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? sm.red[0][tt][e] : -INFINITY;
      }
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < NV; ++i) m = fmaxf(m, v[i]);
      m = warp_max(m);
      float z = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) z += (lane + 32 * i < E) ? expf(v[i] - m) : 0.f;
      z = warp_sum(z);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          const float p = expf(v[i] - m) / z;
          const float dl = p * (dsel[warp][e] - s);
          a.dlogits[(size_t)t * E + e] = dl;
          dbw[warp][e] += dl;
        }
      }
    }
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    float acc = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) acc += dbw[w][e];
    a.db_part[(size_t)blockIdx.x * E + e] = acc;
  }
}

// Router backward, part 1, from the logits the layer forward kept: no second pass over x.  Per
// token, with s = sum_j dg_j g_j:
//   gates not renormalised: p = softmax(logits), dl_e = p_e (dg_slot(e) [e selected] - s);
//   renormalised:           dl_{idx_j} = g_j (dg_j - s), 0 elsewhere (the logits are not read).
// Outputs: dl in fp32 [T, E], as the bf16 operand row [T, Ep] of the dW_r and dx products (zero
// past E), and one db partial per 32 tokens.  A block takes 32 tokens, four per warp; G = min(32,
// EB) lanes share a token, lane i of a group holding experts i, i + G, ... and (k <= G) slot i of
// the token; the group's max and sum are xor shuffles within it.  Every load of a warp's four
// tokens is issued before the arithmetic of the first, so their latencies overlap; what remains
// bounds the kernel by instruction issue.  db: each lane adds its tokens in order, then one thread
// per expert adds the groups in (warp, group) order -- a fixed order.
template <int EB>
__global__ void __launch_bounds__(kThreads)
    router_dlogits_saved_kernel(RouterBwdArgs a, const float* __restrict__ logits, uint16_t* __restrict__ dl_bf16,
                                int T, int E, int Ep, int k, int renorm) {
  constexpr int G = EB < 32 ? EB : 32;   // lanes per token
  constexpr int TPW = 32 / G;            // tokens per warp pass
  constexpr int NV = EB / G;             // experts per lane
  constexpr int kTokens = 32;            // tokens per block (one db partial)
  constexpr int kWarps = kThreads / 32;
  constexpr int kPerWarp = kTokens / kWarps;
  constexpr int P = kPerWarp / TPW;      // passes per warp
  static_assert(kPerWarp % TPW == 0, "whole passes per warp");
  __shared__ float red[kWarps * TPW * EB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / G, li = lane % G, g0 = lane - li;
  const bool slots_in_lanes = k <= G;    // else each lane walks the token's slots itself
  // every pass's loads first (rows past T load nothing; every lane runs every pass, since the
  // shuffles below take the whole warp)
  int sid[P];
  float sg[P], sdg[P], lv[P][NV];
#pragma unroll
  for (int ps = 0; ps < P; ++ps) {
    const int t = blockIdx.x * kTokens + warp * kPerWarp + ps * TPW + grp;
    const bool live = t < T;
    sid[ps] = -1;
    sg[ps] = sdg[ps] = 0.f;
    if (live && slots_in_lanes && li < k) {
      sid[ps] = a.idx[(size_t)t * k + li];
      sg[ps] = a.gates[(size_t)t * k + li];
      sdg[ps] = a.dgates[(size_t)t * k + li];
    }
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = li + G * i;
      lv[ps][i] = (!renorm && live && e < E) ? logits[(size_t)t * E + e] : -INFINITY;
    }
  }
  float dbacc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) dbacc[i] = 0.f;
#pragma unroll
  for (int ps = 0; ps < P; ++ps) {
    const int t = blockIdx.x * kTokens + warp * kPerWarp + ps * TPW + grp;
    const bool live = t < T;
    const int tl = live ? t : 0;
    float s = 0.f;
    float dsel[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) dsel[i] = 0.f;
    if (slots_in_lanes) {
      // s by an xor tree inside the group (lanes past k hold zeros); then each slot's share of dl,
      // formed by the lane that holds it, goes to every lane of the group with its expert
      s = sdg[ps] * sg[ps];
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      const float vmine = renorm ? sg[ps] * (sdg[ps] - s) : sdg[ps];
      for (int j = 0; j < k; ++j) {
        const int e = __shfl_sync(0xffffffffu, sid[ps], g0 + j);
        const float v = __shfl_sync(0xffffffffu, vmine, g0 + j);
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (e == li + G * i) dsel[i] += v;
      }
    } else {
      for (int j = 0; j < k; ++j) s += a.dgates[(size_t)tl * k + j] * a.gates[(size_t)tl * k + j];
      for (int j = 0; j < k; ++j) {
        const int e = a.idx[(size_t)tl * k + j];
        const float dg = a.dgates[(size_t)tl * k + j];
        const float v = renorm ? a.gates[(size_t)tl * k + j] * (dg - s) : dg;
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (e == li + G * i) dsel[i] += v;
      }
    }
    float dl[NV];
    if (renorm) {
#pragma unroll
      for (int i = 0; i < NV; ++i) dl[i] = li + G * i < E ? dsel[i] : 0.f;
    } else {
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < NV; ++i) m = fmaxf(m, lv[ps][i]);
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      // the fast exponential and one reciprocal a token: the kernel is bound by instruction issue,
      // and dl feeds bf16 products and fp32 sums held to the bf16 gradient rule
      float ex[NV], z = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        ex[i] = li + G * i < E ? __expf(lv[ps][i] - m) : 0.f;
        z += ex[i];
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
      const float rz = 1.f / z;
#pragma unroll
      for (int i = 0; i < NV; ++i) dl[i] = li + G * i < E ? ex[i] * rz * (dsel[i] - s) : 0.f;
    }
    if (!live) continue;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = li + G * i;
      if (e < E) a.dlogits[(size_t)t * E + e] = dl[i];
      if (e < Ep) dl_bf16[(size_t)t * Ep + e] = (uint16_t)(pack_bf16(dl[i], 0.f) & 0xFFFFu);
      dbacc[i] += dl[i];
    }
    // columns [EB, Ep) of the bf16 row are zero (EB < Ep only for E <= 32: 16-byte pieces)
    for (int c = EB + 8 * li; c < Ep; c += 8 * G)
      *reinterpret_cast<uint4*>(dl_bf16 + (size_t)t * Ep + c) = make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) red[(warp * TPW + grp) * EB + li + G * i] = dbacc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    float v = 0.f;
    for (int r = 0; r < kWarps * TPW; ++r) v += red[r * EB + e];
    a.db_part[(size_t)blockIdx.x * E + e] = v;
  }
}

// Router backward, part 3: fixed-order sums of the dW_r and db partials.  The first dw_blocks
// blocks sum dW_r element by element over the splits; then one warp per expert sums its db
// partials, lane l taking blocks l, l + 32, ... and a shuffle tree of fixed shape joining the lanes
// (the partials of the bias run to thousands of blocks: a single thread's chain would dominate).
__global__ void router_reduce_kernel(RouterBwdArgs a, int d, int E, int nsplit, int nblk, int dw_blocks) {
  if ((int)blockIdx.x < dw_blocks) {
    const size_t n = (size_t)d * E;
    for (size_t p = blockIdx.x * (size_t)blockDim.x + threadIdx.x; p < n; p += (size_t)dw_blocks * blockDim.x) {
      float v = 0.f;
      for (int s = 0; s < nsplit; ++s) v += a.dwr_part[(size_t)s * n + p];
      a.dW_r[p] = v;
    }
    return;
  }
  const int e = ((int)blockIdx.x - dw_blocks) * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (a.db_r == nullptr || e >= E) return;
  float v = 0.f;
  for (int b = lane; b < nblk; b += 32) v += a.db_part[(size_t)b * E + e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  if (lane == 0) a.db_r[e] = v;
}

int bucket_of(int E) {
  int b = 8;
  while (b < E) b *= 2;
  return b;
}

template <int EB>
cudaError_t route_fwd_eb(const Cfg& c, const RouteArgs& a, cudaStream_t s) {
  using S = RouteShape<EB>;
  const size_t smem = sizeof(LogitSmem<EB>);
  auto kern = route_fwd_kernel<EB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = (c.T + S::BT - 1) / S::BT;
  prof_mark(kKRoute, s, true);
  kern<<<grid, kThreads, smem, s>>>(a, c.T, c.d, c.E, c.k, c.renorm);
  prof_mark(kKRoute, s, false);
  return cudaGetLastError();
}

template <int EB>
cudaError_t router_dlogits_eb(const Cfg& c, const Layout& L, const RouterBwdArgs& a, cudaStream_t s) {
  const size_t smem = sizeof(LogitSmem<EB>);
  auto kern = router_dlogits_kernel<EB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_mark(kKRouterDlogits, s, true);
  kern<<<L.nblk_router, kThreads, smem, s>>>(a, c.T, c.d, c.E, c.k, c.renorm);
  prof_mark(kKRouterDlogits, s, false);
  return cudaGetLastError();
}

// W_r [d, E] fp32 -> three bf16 parts, K-major [3][Ep][d]: hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid) (each difference is exact in fp32), so hi + mid + lo equals w to within
// fp32 rounding; experts E..Ep-1 are zero.  32 x 32 tiles transposed through shared memory.
__global__ void split_wr_kernel(const float* __restrict__ W_r, int d, int E, int Ep, uint16_t* __restrict__ wr3) {
  __shared__ float tile[32][33];
  const int r0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, e = e0 + tx;
    tile[i][tx] = (r < d && e < E) ? W_r[(size_t)r * E + e] : 0.f;
  }
  __syncthreads();
  const size_t n = (size_t)Ep * d;
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i, r = r0 + tx;
    if (e >= Ep || r >= d) continue;
    const float w = tile[tx][i];
    const uint32_t hi = pack_bf16(w, 0.f) & 0xFFFFu;
    const float r1 = w - bf16_lo(hi);
    const uint32_t mid = pack_bf16(r1, 0.f) & 0xFFFFu;
    const float r2 = r1 - bf16_lo(mid);
    const uint32_t lo = pack_bf16(r2, 0.f) & 0xFFFFu;
    const size_t o = (size_t)e * d + r;
    wr3[o] = (uint16_t)hi;
    wr3[n + o] = (uint16_t)mid;
    wr3[2 * n + o] = (uint16_t)lo;
  }
}

// dst[r][c] = bf16(src[r][c]) for c < cols, 0 for cols <= c < ld (rows of the tensor-core operands)
__global__ void to_bf16_rows_kernel(const float* __restrict__ src, int rows, int cols, int ld,
                                    uint16_t* __restrict__ dst) {
  const size_t n = (size_t)rows * ld;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / ld;
    const int c = (int)(i - r * ld);
    const float v = c < cols ? src[r * cols + c] : 0.f;
    dst[i] = (uint16_t)(pack_bf16(v, 0.f) & 0xFFFFu);
  }
}

}  // namespace

// blocks (and db partials) of router_dlogits_saved_kernel: 32 tokens each
int router_saved_blocks(const Cfg& c) { return (c.T + 31) / 32; }

int route_block_tokens(int E) {
  switch (bucket_of(E)) {
    case 8: return RouteShape<8>::BT;
    case 16: return RouteShape<16>::BT;
    case 32: return RouteShape<32>::BT;
    case 64: return RouteShape<64>::BT;
    case 128: return RouteShape<128>::BT;
    default: return RouteShape<256>::BT;
  }
}

cudaError_t launch_route(const Cfg& c, const RouteArgs& a, cudaStream_t s) {
  switch (bucket_of(c.E)) {
    case 8: return route_fwd_eb<8>(c, a, s);
    case 16: return route_fwd_eb<16>(c, a, s);
    case 32: return route_fwd_eb<32>(c, a, s);
    case 64: return route_fwd_eb<64>(c, a, s);
    case 128: return route_fwd_eb<128>(c, a, s);
    default: return route_fwd_eb<256>(c, a, s);
  }
}

cudaError_t launch_router_dlogits(const Cfg& c, const Layout& L, const RouterBwdArgs& a, cudaStream_t s) {
  switch (bucket_of(c.E)) {
    case 8: return router_dlogits_eb<8>(c, L, a, s);
    case 16: return router_dlogits_eb<16>(c, L, a, s);
    case 32: return router_dlogits_eb<32>(c, L, a, s);
    case 64: return router_dlogits_eb<64>(c, L, a, s);
    case 128: return router_dlogits_eb<128>(c, L, a, s);
    default: return router_dlogits_eb<256>(c, L, a, s);
  }
}

template <int EB>
cudaError_t router_dlogits_saved_eb(const Cfg& c, const Layout& L, const RouterBwdArgs& a, const float* logits,
                                    uint16_t* dl_bf16, cudaStream_t s) {
  prof_mark(kKRouterDlogits, s, true);
  router_dlogits_saved_kernel<EB><<<router_saved_blocks(c), kThreads, 0, s>>>(a, logits, dl_bf16, c.T, c.E, L.Ep, c.k,
                                                                              c.renorm);
  prof_mark(kKRouterDlogits, s, false);
  return cudaGetLastError();
}

cudaError_t launch_router_dlogits_saved(const Cfg& c, const Layout& L, const RouterBwdArgs& a, const float* logits,
                                        uint16_t* dl_bf16, cudaStream_t s) {
  if (!c.renorm && logits == nullptr) return cudaErrorInvalidValue;
  switch (bucket_of(c.E)) {
    case 8: return router_dlogits_saved_eb<8>(c, L, a, logits, dl_bf16, s);
    case 16: return router_dlogits_saved_eb<16>(c, L, a, logits, dl_bf16, s);
    case 32: return router_dlogits_saved_eb<32>(c, L, a, logits, dl_bf16, s);
    case 64: return router_dlogits_saved_eb<64>(c, L, a, logits, dl_bf16, s);
    case 128: return router_dlogits_saved_eb<128>(c, L, a, logits, dl_bf16, s);
    default: return router_dlogits_saved_eb<256>(c, L, a, logits, dl_bf16, s);
  }
}

cudaError_t launch_router_reduce(const Cfg& c, const Layout& L, const RouterBwdArgs& a, int nblk, cudaStream_t s) {
  const size_t n = (size_t)c.d * c.E;
  const int dw_blocks = (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 4));
  const int db_blocks = a.db_r != nullptr ? (c.E + 7) / 8 : 0;   // 8 warps, one expert each
  prof_mark(kKRouterReduce, s, true);
  router_reduce_kernel<<<dw_blocks + db_blocks, 256, 0, s>>>(a, c.d, c.E, L.nsplit_dwr, nblk, dw_blocks);
  prof_mark(kKRouterReduce, s, false);
  return cudaGetLastError();
}

bool router_on_tensor_cores(const Cfg& c) { return c.E <= 128 && c.k <= 8; }
bool router_bwd_on_tensor_cores(const Cfg& c) { return router_on_tensor_cores(c) && !c.renorm; }

cudaError_t launch_split_wr(const float* W_r, int d, int E, int Ep, uint16_t* wr3, cudaStream_t s) {
  const dim3 grid((d + 31) / 32, (Ep + 31) / 32);
  prof_mark(kKSplitWr, s, true);
  split_wr_kernel<<<grid, 256, 0, s>>>(W_r, d, E, Ep, wr3);
  prof_mark(kKSplitWr, s, false);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16_rows(const float* src, int rows, int cols, int ld, uint16_t* dst, cudaStream_t s) {
  const size_t n = (size_t)rows * ld;
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8));
  prof_mark(kKToBf16, s, true);
  to_bf16_rows_kernel<<<blocks, 256, 0, s>>>(src, rows, cols, ld, dst);
  prof_mark(kKToBf16, s, false);
  return cudaGetLastError();
}

}  // namespace moe
