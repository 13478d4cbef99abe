// Router logits for narrow routers (E <= 32, k <= 8) on the tensor cores, streaming x once at the
// HBM rate: logits = x W_r (+ b), softmax, top-k and gates (forward), or the router's dlogits
// (backward, gates not renormalised).  Sources: the Piper explainer ("the problem": a router sends
// each token to a few experts), the MoEBlaze summary (Limitations: static top-k routing); the
// formulas are the plain softmax-then-top-k reading.
//
// With few experts the logits are a thin product: x [T, d] bf16 is read once (T d 2 bytes) for
// 2 T d E FLOP, so the kernel is bound by HBM, and the whole GPU has to stream x.  Design:
//   * W_r (fp32) is split into three bf16 parts hi + mid + lo (each difference exact in fp32), so
//     every partial product with the bf16 x is exact and only the fp32 accumulation rounds.  The
//     parts are stacked along the MMA's N dimension -- rows [0, EB) hi, [EB, 2EB) mid, [2EB, 3EB)
//     lo, with EB = E rounded up to 8, 16 or 32 -- so one tcgen05.mma (M = 128 tokens,
//     N = 3 EB rounded up to 16, K = 16) covers all three.
//   * A tensor-core accumulator loses about one fp32 unit of its own size per K step, so K runs in
//     256-wide slices (16 steps); each slice starts a fresh accumulator, and the epilogue adds
//     hi + (mid + lo) of every slice into fp32 registers, one token per TMEM lane.
//   * The (tile, slice) pairs, tiles outer, are cut into kRanges contiguous ranges of equal
//     length (to one slice), one per CTA, so every SM streams the same share of x even when T / 128
//     is below the SM count (8192 tokens: 64 tiles of 16 slices, about 6.7 slices a CTA).  A CTA
//     sums its slices of one tile in registers; when a tile is split between CTAs, each writes its
//     share (a segment) as partial logits, and per 32-token quarter of the tile a counter finds the
//     last segment to finish: that warp sums the segments in range order (deterministic, whichever
//     CTA finishes last) and runs the selection (forward) or dlogits (backward).  A tile covered by
//     one CTA is finished from registers.
// Warp roles: warp 0 issues TMA loads of x and of the stacked W_r parts into a ring of stages,
// warp 1 (one thread) issues the MMAs, warps 2-5 are the epilogue (TMEM lane quarters).  Every
// wait is bounded (MOE_ERR_TIMEOUT instead of a hang).
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {

namespace {

constexpr int kTok = 128;                          // tokens per tile (TMEM lanes)
constexpr int kKB = 64;                            // K block: 64 bf16 = one 128-byte swizzle row
constexpr int kSliceKB = 4;                        // K blocks per accumulator slice (K = 256)
constexpr uint32_t kXBytes = kTok * kKB * 2;       // 16 KB of x per stage
constexpr int kThreads = 192;                      // producer, MMA, four epilogue warps
constexpr uint32_t kStageBudget = 212 * 1024;      // shared memory for the stage ring
constexpr int kRanges = 152;                       // slice ranges: one CTA each (152 SMs)
constexpr int kTopK = 8;

struct Params {
  CUtensorMap tmX, tmW;
  const float* b_r;
  int T, d, E, k, renorm;
  int nkb, nslice;                   // K blocks and 256-wide slices of d_model
  long long nsl;                     // (tile, slice) pairs: ntiles * nslice
  int nranges, maxseg;               // CTAs (ranges) and the most segments a tile has
  float* part;                       // [ntiles][maxseg][EB][128] partial logits of split tiles
  uint32_t* cnt;                     // [ntiles][4] segments finished per token quarter
  int32_t* idx; float* gates; float* logits;                       // forward
  const float* dgates; float* dlogits; uint16_t* dl_bf16;          // backward (idx, gates read)
  float* db_part;                    // backward: [ntiles * 4][E]
  Hdr* hdr;
};

template <int EB>
struct Shape {
  static constexpr int kNb = (3 * EB + 15) / 16 * 16;             // MMA N: stacked parts, padded
  static constexpr uint32_t kWBytes = kNb * kKB * 2;
  static constexpr uint32_t kStageBytes = kXBytes + kWBytes;      // multiple of 1024
  static constexpr int kStages = (int)std::min<uint32_t>(10, kStageBudget / kStageBytes);
  static constexpr int kPieces = (kNb + 31) / 32;                 // 32-column TMEM loads per slice
  static constexpr int kAccBufs = kNb <= 128 ? 4 : 2;             // accumulators in 512 TMEM columns
  static constexpr uint32_t kAccStride = 512 / kAccBufs;
  static constexpr int kSegBatch = EB <= 8 ? 4 : (EB <= 16 ? 2 : 1);   // segments loaded at once
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 256;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-aligned");
  static_assert(8 * (2 * kStages + 2 * kAccBufs + 1) + 8 <= 256, "barriers fit their 256 bytes");
  static_assert(kSmem <= 232448, "shared memory per block");
};

// Range b covers (tile, slice) pairs [first(b), first(b + 1)), first(b) = floor(b nsl / nranges);
// the range holding pair s is the last b with first(b) <= s.
__host__ __device__ __forceinline__ long long range_first(long long b, long long nsl, int nranges) {
  return b * nsl / nranges;
}
__host__ __device__ __forceinline__ int range_of(long long s, long long nsl, int nranges) {
  return (int)(((s + 1) * nranges - 1) / nsl);
}

// Atomic add with acquire-release semantics at GPU scope: publishes the writes this thread has
// observed (the warp's, after __syncwarp) and sees those published before it by other CTAs.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float warp_sum32(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Softmax, top-k (larger logit first, a tie keeping the lower expert index) and gates of one
// token (forward), or its dlogits (backward, not renormalised).  l[] holds the logits (bias
// added); `live` is false for the rows of the last tile past T.
template <int EB, bool kBwd>
__device__ __forceinline__ void finish_token(const Params& p, const float (&l)[EB], int t, bool live, int tile,
                                             int q, int lane) {
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EB; ++e)
    if (e < p.E) m = fmaxf(m, l[e]);
  float z = 0.f;
#pragma unroll
  for (int e = 0; e < EB; ++e)
    if (e < p.E) z += expf(l[e] - m);
  if (!kBwd) {
    if (!live) return;
    float tv[kTopK];
    int ti[kTopK];
#pragma unroll
    for (int s = 0; s < kTopK; ++s) {
      tv[s] = -INFINITY;
      ti[s] = 0x7fffffff;
    }
    if (p.logits != nullptr) {   // 16-byte stores when the rows are 16-byte aligned (E a multiple of 4)
      float* row = p.logits + (size_t)t * p.E;
      if ((p.E & 3) == 0) {
#pragma unroll
        for (int q = 0; q < EB / 4; ++q)
          if (4 * q < p.E) *reinterpret_cast<float4*>(row + 4 * q) = make_float4(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < EB; ++e)
          if (e < p.E) row[e] = l[e];
      }
    }
#pragma unroll
    for (int e = 0; e < EB; ++e) {
      if (e >= p.E) continue;
      float cv = l[e];
      int ci = e;
#pragma unroll
      for (int s = 0; s < kTopK; ++s)
        if (cv > tv[s]) {
          const float fv = tv[s];
          const int fi = ti[s];
          tv[s] = cv;
          ti[s] = ci;
          cv = fv;
          ci = fi;
        }
    }
    float zsel = 0.f;
#pragma unroll
    for (int s = 0; s < kTopK; ++s)
      if (s < p.k) zsel += expf(tv[s] - m);
    const float denom = p.renorm ? zsel : z;
#pragma unroll
    for (int s = 0; s < kTopK; ++s)
      if (s < p.k) {
        p.idx[(size_t)t * p.k + s] = ti[s];
        p.gates[(size_t)t * p.k + s] = expf(tv[s] - m) / denom;
      }
    return;
  }
  // backward: dl_e = p_e (dg_slot(e) [e selected] - sum_j dg_j g_j)
  float sdg = 0.f;
  int sid[kTopK];
  float sgd[kTopK];
#pragma unroll
  for (int s = 0; s < kTopK; ++s) {
    sid[s] = -1;
    sgd[s] = 0.f;
    if (live && s < p.k) {
      sid[s] = p.idx[(size_t)t * p.k + s];
      sgd[s] = p.dgates[(size_t)t * p.k + s];
      sdg += sgd[s] * p.gates[(size_t)t * p.k + s];
    }
  }
  float dl[EB];
#pragma unroll
  for (int e = 0; e < EB; ++e) {
    float dsel = 0.f;
#pragma unroll
    for (int s = 0; s < kTopK; ++s) dsel += (sid[s] == e) ? sgd[s] : 0.f;
    dl[e] = (live && e < p.E) ? expf(l[e] - m) / z * (dsel - sdg) : 0.f;
  }
  if (live) {
#pragma unroll
    for (int e = 0; e < EB; ++e)
      if (e < p.E) p.dlogits[(size_t)t * p.E + e] = dl[e];
    // the bf16 operand row of the dW_r and dx products: 64 columns (E <= 32), zero past E
    uint4* row = reinterpret_cast<uint4*>(p.dl_bf16 + (size_t)t * 64);
#pragma unroll
    for (int c = 0; c < 64; c += 8) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int e0 = c + 2 * h, e1 = e0 + 1;
        w[h] = pack_bf16(e0 < EB ? dl[e0 < EB ? e0 : 0] : 0.f, e1 < EB ? dl[e1 < EB ? e1 : 0] : 0.f);
      }
      row[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  // db partial of these 32 tokens (one per expert, summed over the warp in a fixed order)
#pragma unroll
  for (int e = 0; e < EB; ++e) {
    const float v = warp_sum32(dl[e]);
    if (lane == 0 && e < p.E) p.db_part[((size_t)tile * 4 + q) * p.E + e] = v;
  }
}

template <int EB, bool kBwd>
__global__ void __launch_bounds__(kThreads, 1) route_stream_kernel(const __grid_constant__ Params p) {
  using S = Shape<EB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)S::kStages * S::kStageBytes);
  uint64_t* empty = full + S::kStages;
  uint64_t* tfull = empty + S::kStages;
  uint64_t* tempty = tfull + S::kAccBufs;
  uint64_t* drain = tempty + S::kAccBufs;   // the MMA thread's last commit, waited for before TMEM is freed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's (tile, slice) pairs, tiles outer
  const long long sl0 = range_first(blockIdx.x, p.nsl, p.nranges);
  const long long sl1 = range_first(blockIdx.x + 1, p.nsl, p.nranges);
  // the producer's position (thread 0): the next (tile, slice) pair, its next K block and stage
  long long lsp = sl0;
  int lkb = (int)(sl0 % p.nslice) * kSliceKB;
  int stage = 0, uses = 0;
  uint32_t phase = 0;
  auto issue = [&]() {   // one stage's loads at the producer's position, then step past it
    const int tile = (int)(lsp / p.nslice), sl = (int)(lsp - (long long)tile * p.nslice);
    uint8_t* st = stages + (size_t)stage * S::kStageBytes;
    mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
    tma_load_2d(st, &p.tmX, &full[stage], lkb * kKB, tile * kTok);
    tma_load_2d(st + kXBytes, &p.tmW, &full[stage], lkb * kKB, 0);
    ++uses;
    if (++stage == S::kStages) {
      stage = 0;
      phase ^= 1;
    }
    if (++lkb >= min(p.nkb, (sl + 1) * kSliceKB)) {
      ++lsp;
      lkb = (int)(lsp % p.nslice) * kSliceKB;
    }
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < S::kAccBufs; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch(&p.tmX);
    tma_prefetch(&p.tmW);
    // a fresh ring needs no wait: the first stages' loads leave before the block's setup (TMEM
    // allocation, the barrier), so that the setup overlaps their trip to memory
    while (uses < S::kStages && lsp < sl1) issue();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t limit = wait_limit_ns(p.hdr);

  if (warp == 0) {
    if (lane == 0) {
      while (lsp < sl1 && !*abort_flag) {
        if (!mbar_wait(&empty[stage], phase ^ 1, limit, abort_flag)) {
          record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmProducer);
          *abort_flag = 1;
          break;
        }
        issue();
      }
      // every load this CTA issued lands before its shared memory is released (bounded)
      drain_fills(full, S::kStages, stage, phase, uses, limit);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kTok, S::kNb, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (long long sp = sl0; sp < sl1 && ok && !*abort_flag; ++sp) {
        const int sl = (int)(sp % p.nslice);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, limit, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + (uint32_t)acc * S::kAccStride;
        const int kb0 = sl * kSliceKB, kb1 = min(p.nkb, kb0 + kSliceKB);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, limit, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + (size_t)stage * S::kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            umma_bf16(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kXBytes + kk * 32), idesc,
                      (kb != kb0 || kk != 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == S::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == S::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) {
        record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmMma);
        *abort_flag = 1;
      }
      // every MMA this thread issued has completed before TMEM is freed (bounded)
      umma_commit(drain);
      mbar_wait_drain(drain, 0, limit);
    }
  } else {
    const int q = warp & 3;              // TMEM lane quarter of this warp
    const int row = q * 32 + lane;       // token within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    float l[EB];
#pragma unroll
    for (int e = 0; e < EB; ++e) l[e] = 0.f;
    for (long long sp = sl0; sp < sl1; ++sp) {
      const int tile = (int)(sp / p.nslice);
      if (!mbar_wait_idle(&tfull[acc], acc_phase, limit, abort_flag)) {
        record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem_base + (uint32_t)acc * S::kAccStride + ((uint32_t)(q * 32) << 16);
      // columns j = part * EB + e; pieces go from the last (lo) to the first (hi) so that each
      // expert's slice sum is hi + (mid + lo)
      float mlo[EB];
#pragma unroll
      for (int c = S::kPieces - 1; c >= 0; --c) {
        uint32_t v[32];
        tmem_ld32(ta + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 31; i >= 0; --i) {
          const int j = c * 32 + i;
          if (j >= 3 * EB) continue;
          const int part = j / EB, e = j % EB;
          const float x = __uint_as_float(v[i]);
          if (part == 2) mlo[e] = x;
          else if (part == 1) mlo[e] += x;
          else l[e] += x + mlo[e];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == S::kAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
      // the tile's slices in this range end here: emit its sums
      if (sp + 1 < sl1 && (sp + 1) / p.nslice == tile) continue;
      const int t = tile * kTok + row;
      const bool live = t < p.T;
      const long long first = (long long)tile * p.nslice;
      const int b0 = range_of(first, p.nsl, p.nranges);
      const int nseg = range_of(first + p.nslice - 1, p.nsl, p.nranges) - b0 + 1;
      if (nseg > 1) {
        // publish this CTA's segment; the quarter's last segment to arrive sums all of them
        float* mine = p.part + ((size_t)(tile * p.maxseg + ((int)blockIdx.x - b0)) * EB) * kTok + row;
#pragma unroll
        for (int e = 0; e < EB; ++e) mine[(size_t)e * kTok] = l[e];
        // the warp's stores, then one release/acquire count: the last segment's warp sees every
        // segment written before its count
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(&p.cnt[tile * 4 + q], 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
#pragma unroll
        for (int e = 0; e < EB; ++e) l[e] = 0.f;
        if (old != (uint32_t)(nseg - 1)) continue;
        __syncwarp();   // orders the lanes' loads below after lane 0's acquire
        // sum the segments in range order, kSegBatch segments' loads in flight at a time
        const float* base = p.part + (size_t)tile * p.maxseg * EB * kTok + row;
        for (int sg0 = 0; sg0 < nseg; sg0 += S::kSegBatch) {
          float v[S::kSegBatch][EB];
#pragma unroll
          for (int b = 0; b < S::kSegBatch; ++b)
#pragma unroll
            for (int e = 0; e < EB; ++e)
              v[b][e] = sg0 + b < nseg ? __ldcg(base + ((size_t)(sg0 + b) * EB + e) * kTok) : 0.f;
#pragma unroll
          for (int b = 0; b < S::kSegBatch; ++b)
            if (sg0 + b < nseg) {
#pragma unroll
              for (int e = 0; e < EB; ++e) l[e] += v[b][e];
            }
        }
      }
#pragma unroll
      for (int e = 0; e < EB; ++e)
        if (p.b_r != nullptr && e < p.E) l[e] += __ldg(p.b_r + e);
      finish_token<EB, kBwd>(p, l, t, live, tile, q, lane);
#pragma unroll
      for (int e = 0; e < EB; ++e) l[e] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// W_r [d, E] fp32 -> the stacked bf16 parts [Nb][d] (K-major): row part * EB + e holds part
// `part` of column e of W_r (hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid), each
// difference exact in fp32); rows of experts >= E and rows >= 3 EB are zero.  Also zeroes the
// per-quarter part counters of the router kernel that follows on the same stream.
__global__ void split_wr_stack_kernel(const float* __restrict__ W_r, int d, int E, int EB, int Nb,
                                      uint16_t* __restrict__ ws, uint32_t* __restrict__ cnt, int ncnt) {
  const size_t n = (size_t)Nb * d;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n + ncnt;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i >= n) {
      cnt[i - n] = 0u;
      continue;
    }
    const int r = (int)(i / d), k = (int)(i - (size_t)r * d);
    const int part = r / EB, e = r - part * EB;
    uint32_t out = 0;
    if (part < 3 && e < E) {
      const float w = W_r[(size_t)k * E + e];
      const uint32_t hi = pack_bf16(w, 0.f) & 0xFFFFu;
      const float r1 = w - bf16_lo(hi);
      const uint32_t mid = pack_bf16(r1, 0.f) & 0xFFFFu;
      const float r2 = r1 - bf16_lo(mid);
      const uint32_t lo = pack_bf16(r2, 0.f) & 0xFFFFu;
      out = part == 0 ? hi : (part == 1 ? mid : lo);
    }
    ws[i] = (uint16_t)out;
  }
}

int bucket_eb(int E) { return E <= 8 ? 8 : (E <= 16 ? 16 : 32); }

template <int EB, bool kBwd>
cudaError_t launch_eb(const Cfg& c, const Layout& L, const RouterStreamArgs& a, cudaStream_t s) {
  using S = Shape<EB>;
  const RouterStreamPlan pl = router_stream_plan(c);
  if (L.Ep != 64) return cudaErrorInvalidValue;   // the bf16 dlogits rows are 64 wide for E <= 32
  Params p{};
  if (!map_2d(&p.tmX, a.x, c.d, c.T, 64, 128) || !map_2d(&p.tmW, a.wstack, c.d, S::kNb, 64, S::kNb))
    return cudaErrorInvalidValue;
  p.b_r = a.b_r;
  p.T = c.T;
  p.d = c.d;
  p.E = c.E;
  p.k = c.k;
  p.renorm = c.renorm;
  p.nkb = c.d / kKB;
  p.nslice = pl.nslice;
  p.nsl = (long long)pl.ntiles * pl.nslice;
  p.nranges = pl.nranges;
  p.maxseg = pl.maxseg;
  p.part = a.part;
  p.cnt = a.cnt;
  p.idx = a.idx;
  p.gates = a.gates;
  p.logits = a.logits;
  p.dgates = a.dgates;
  p.dlogits = a.dlogits;
  p.dl_bf16 = a.dl_bf16;
  p.db_part = a.db_part;
  p.hdr = a.hdr;
  auto kern = route_stream_kernel<EB, kBwd>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kSmem);
  if (e != cudaSuccess) return e;
  const int grid = p.nranges;
  prof_mark(kBwd ? kKRouterDlogits : kKRoute, s, true);
  kern<<<grid, kThreads, S::kSmem, s>>>(p);
  prof_mark(kBwd ? kKRouterDlogits : kKRoute, s, false);
  return cudaGetLastError();
}

template <bool kBwd>
cudaError_t launch_stream(const Cfg& c, const Layout& L, const RouterStreamArgs& a, cudaStream_t s) {
  const int EB = bucket_eb(c.E);
  const int Nb = (3 * EB + 15) / 16 * 16;
  const RouterStreamPlan pl = router_stream_plan(c);
  const int ncnt = pl.ntiles * 4;
  const size_t n = (size_t)Nb * c.d + ncnt;
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 4));
  prof_mark(kKSplitWr, s, true);
  split_wr_stack_kernel<<<blocks, 256, 0, s>>>(a.W_r, c.d, c.E, EB, Nb, a.wstack, a.cnt, ncnt);
  prof_mark(kKSplitWr, s, false);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (EB) {
    case 8: return launch_eb<8, kBwd>(c, L, a, s);
    case 16: return launch_eb<16, kBwd>(c, L, a, s);
    default: return launch_eb<32, kBwd>(c, L, a, s);
  }
}

}  // namespace

// Up to 32 experts.  Wider routers stay on the tensor-core kernel that gives each 128-token tile
// one CTA (gemm.cu): at E = 64 the stacked parts (192 rows) make each stage 40 KB for 16 KB of x,
// and halving the x bytes in flight cost more than the split K gains (measured, T = 16384,
// d = 2048, L2 cold: 62 against 39 us forward, 95 against 46 us for the dlogits pass).
bool router_stream_eligible(const Cfg& c) { return c.E <= 32 && c.k <= kTopK; }

// kRanges CTAs (fewer when there are fewer (tile, slice) pairs), each a contiguous run of pairs;
// maxseg = the most ranges one tile is split between (sizes the partial-logit buffer).  Fixed by
// the configuration alone, so the summation order does not depend on the device.
RouterStreamPlan router_stream_plan(const Cfg& c) {
  RouterStreamPlan pl{};
  pl.ntiles = (c.T + kTok - 1) / kTok;
  pl.nslice = (c.d / kKB + kSliceKB - 1) / kSliceKB;
  const long long nsl = (long long)pl.ntiles * pl.nslice;
  pl.nranges = (int)std::min<long long>(kRanges, nsl);
  pl.maxseg = 1;
  for (int t = 0; t < pl.ntiles; ++t) {
    const long long first = (long long)t * pl.nslice;
    const int nseg = range_of(first + pl.nslice - 1, nsl, pl.nranges) - range_of(first, nsl, pl.nranges) + 1;
    pl.maxseg = std::max(pl.maxseg, nseg);
  }
  pl.eb = bucket_eb(c.E);
  return pl;
}

cudaError_t launch_route_stream(const Cfg& c, const Layout& L, const RouterStreamArgs& a, cudaStream_t s) {
  return launch_stream<false>(c, L, a, s);
}

cudaError_t launch_router_dlogits_stream(const Cfg& c, const Layout& L, const RouterStreamArgs& a,
                                         cudaStream_t s) {
  return launch_stream<true>(c, L, a, s);
}

}  // namespace moe
