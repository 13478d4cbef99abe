// Dispatch queues (MoEBlaze, Methodology item 1): tokens reach their experts through per-expert
// queues built on the fly -- a histogram, an exclusive prefix sum and a stable permutation --
// instead of a dense token-by-expert routing matrix.
//
// dispatch_scan_kernel: one pass over the T*k assignments in token order.  Each block ranks its
//   4096 assignments per expert (warp match + shared-memory running counts, so ranks follow the
//   (t, j) order), publishes its per-expert aggregate, and finds its per-expert exclusive prefix
//   with a decoupled look-back over the preceding blocks (bounded spin).  The last block to
//   finish builds the routing tables: counts, capacity, exact offsets, 256-row padded segment
//   starts, pad-row prefix and the segment order by size.
// dispatch_gather_kernel: token owner.  A warp reads each x (and dy) row once, 16 bytes per lane,
//   and writes it to every kept slot's row (and every shared expert's row); then zeroes pad rows.
//   Rows are moved as 16-byte vectors, so the FP8 forward gathers e4m3 token rows (d bytes) through
//   the same kernel as rows of d/2 two-byte elements, with their row scales beside them.  For GEMMs
//   that gather their operand rows themselves (tile::gather4 from token order) the kernel moves no
//   data and writes only the tables, the token of every padded row and, for the backward, its gate.
//   For the FP8 backward it also quantises: a token's x and dy rows get their e4m3 row scales from
//   one amax pass, and each vector's codes are written beside its bf16 copy to every expert row,
//   so no pass re-reads the k-fold expert rows to quantise them.
#include <mutex>

#include "common.cuh"
#include "e4m3.cuh"

namespace moe {
namespace {

constexpr int kWarps = kScanThreads / 32;
constexpr int kPerWarp = kScanChunk / kWarps;   // 256 assignments, 8 rounds of 32
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kValueMask = (1u << 30) - 1;

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__global__ void __launch_bounds__(kScanThreads) dispatch_scan_kernel(DispatchArgs a, int N, int T,
                                                                     int E, int S, int C, int nblk,
                                                                     long long row_cap) {
  __shared__ int wcnt[kWarps][kMaxE];   // per-warp running counts, then warp exclusive prefix
  __shared__ int blk_excl[kMaxE];
  __shared__ int s_blk, s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s_blk = (int)atomicAdd(&a.hdr->scan_ticket, 1u);
  for (int i = threadIdx.x; i < kWarps * kMaxE; i += kScanThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const int blk = s_blk;
  const int base = blk * kScanChunk + warp * kPerWarp;

  int my_e[kPerWarp / 32], my_r[kPerWarp / 32];
#pragma unroll
  for (int s = 0; s < kPerWarp / 32; ++s) {
    const int i = base + s * 32 + lane;
    int e = -1;
    if (i < N) {
      e = a.idx[i];
      if (e < 0 || e >= E) {
        record_error(a.hdr, MOE_ERR_BAD_INDEX, kSiteScanIndex);
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int before = (e >= 0) ? wcnt[warp][e] : 0;
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp][e] = before + __popc(peers);
    __syncwarp();
    my_e[s] = e;
    my_r[s] = before + __popc(peers & ((1u << lane) - 1u));
  }
  __syncthreads();

  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int agg = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = agg;
      agg += c;
    }
    uint32_t* st = a.scan_status + (size_t)blk * E + e;
    const bool stall = (blk + 1 == a.hdr->stall_block_p1);
    int excl = 0;
    if (blk == 0) {
      if (!stall) st_release(st, kFlagIncl | (uint32_t)agg);
    } else {
      if (!stall) st_release(st, kFlagAgg | (uint32_t)agg);
      const uint64_t limit = wait_limit_ns(a.hdr);
      const uint64_t t0 = global_ns();
      int b = blk - 1;
      while (b >= 0) {
        const uint32_t v = ld_acquire(a.scan_status + (size_t)b * E + e);
        if ((v & ~kValueMask) == 0) {
          if (global_ns() - t0 > limit) {
            record_error(a.hdr, MOE_ERR_TIMEOUT, kSiteScanLookback);
            break;
          }
          continue;
        }
        excl += (int)(v & kValueMask);
        if ((v & ~kValueMask) == kFlagIncl) break;
        --b;
      }
      if (!stall) st_release(st, kFlagIncl | (uint32_t)((excl + agg) & (int)kValueMask));
    }
    blk_excl[e] = excl;
  }
  __syncthreads();

#pragma unroll
  for (int s = 0; s < kPerWarp / 32; ++s) {
    const int i = base + s * 32 + lane;
    const int e = my_e[s];
    if (i < N && e >= 0) a.rank[i] = blk_excl[e] + wcnt[warp][e] + my_r[s];
  }

  // The last block to finish builds the tables.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&a.hdr->scan_done, 1u) == (unsigned)(nblk - 1));
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  Tables* tb = a.tabs;
  const int G = E + S;
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    const uint32_t v = ld_acquire(a.scan_status + (size_t)(nblk - 1) * E + e);
    const int total = (int)(v & kValueMask);
    tb->counts[e] = total;
    if (a.counts != nullptr) a.counts[e] = total;
    tb->kept[e] = total < C ? total : C;
  } else if (threadIdx.x < G) {
    tb->kept[threadIdx.x] = T;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // A pending device error means the ranks cannot be trusted: publish empty segments so that
    // no later kernel touches rows on their account.
    const bool bad = (*((volatile int*)&a.hdr->status)) != 0;
    int off = 0;
    long long poff = 0, pads = 0;
    for (int g = 0; g < G; ++g) {
      int kept = bad ? 0 : tb->kept[g];
      tb->kept[g] = kept;
      if (g < E) {
        tb->offsets[g] = off;
        if (a.offsets != nullptr) a.offsets[g] = off;
        off += kept;
      }
      const long long padded = ((long long)kept + kRowTile - 1) / kRowTile * kRowTile;
      tb->poff[g] = (int)poff;
      tb->pad_start[g] = (int)pads;
      poff += padded;
      pads += padded - kept;
    }
    tb->offsets[E] = off;
    if (a.offsets != nullptr) a.offsets[E] = off;
    if (poff > row_cap) {   // cannot happen for valid ranks; guard the buffers regardless
      record_error(a.hdr, MOE_ERR_BAD_INDEX, kSiteScanIndex);
      for (int g = 0; g < G; ++g) {
        tb->kept[g] = 0;
        tb->poff[g] = 0;
        tb->pad_start[g] = 0;
      }
      poff = 0;
      pads = 0;
    }
    tb->poff[G] = (int)poff;
    tb->pad_start[G] = (int)pads;
    tb->G = G;
    tb->total_rows = (int)poff;
    tb->n_mtiles = (int)(poff / kRowTile);
    tb->total_pad = (int)pads;
    // every scan block has recorded its errors before counting itself done
    if (a.status_out != nullptr) *a.status_out = *((volatile int*)&a.hdr->status);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    const int pg = tb->poff[g + 1] - tb->poff[g];
    int r = 0;
    for (int h = 0; h < G; ++h) {
      const int ph = tb->poff[h + 1] - tb->poff[h];
      r += (ph > pg) || (ph == pg && h < g);
    }
    tb->seg_order[r] = g;
  }
}

constexpr int kUnroll = 4;   // 16-byte vectors per lane in flight per source row

template <bool kMeta, bool kX, bool kDy, bool kGate, bool kQ = false>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(DispatchArgs a, int T, int k, int E,
                                                              int S, int d) {
  static_assert(!kQ || (kX && kDy), "the quantising gather moves x and dy");
  constexpr bool kGates = kDy || kGate;   // the gate of every padded row
  const Tables* tb = a.tabs;
  const int lane = threadIdx.x & 31;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  const int nvec = d / 8;   // 16-byte pieces per row
  for (int t = gw; t < T; t += nw) {
    const uint4* xs = kX ? reinterpret_cast<const uint4*>(a.x + (size_t)t * d) : nullptr;
    const uint4* dys = kDy ? reinterpret_cast<const uint4*>(a.dy + (size_t)t * d) : nullptr;
    // quant: the token's row scales (amax over the whole row first; the copy pass below re-reads the
    // row from L2) and their reciprocals, warp-uniform
    float sx = 1.f, sd = 1.f, yx = 0.f, yd = 0.f;
    bool rx = true, rd = true;
    if constexpr (kQ) {
      float ax = 0.f, ad = 0.f;
      for (int v = lane; v < nvec; v += 32) {
        ax = fmaxf(ax, amax8_bf16(xs[v]));
        ad = fmaxf(ad, amax8_bf16(dys[v]));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        ax = fmaxf(ax, __shfl_xor_sync(0xffffffffu, ax, off));
        ad = fmaxf(ad, __shfl_xor_sync(0xffffffffu, ad, off));
      }
      sx = e4m3_row_scale(ax);
      sd = e4m3_row_scale(ad);
      rx = e4m3_recip_ok(sx);
      rd = e4m3_recip_ok(sd);
      yx = rx ? __frcp_rn(sx) : 0.f;
      yd = rd ? __frcp_rn(sd) : 0.f;
    }
    for (int jb = 0; jb < k; jb += 32) {
      const int j = jb + lane;
      int prow = -1;
      if (j < k && !kMeta) {
        // tables and rows were built by an earlier dispatch of the same workspace
        const size_t slot = (size_t)t * k + j;
        prow = a.prow_of_slot[slot];
        if (kDy && prow >= 0) a.gate_of_prow[prow] = a.gates[slot];
      } else if (j < k) {
        const size_t slot = (size_t)t * k + j;
        const int e = a.idx[slot];
        const bool valid = e >= 0 && e < E;
        const int r = valid ? a.rank[slot] : 0;
        const bool kept = valid && r >= 0 && r < tb->kept[e];
        prow = kept ? tb->poff[e] + r : -1;
        {
          const int row = kept ? tb->offsets[e] + r : -1;
          if (a.row_of_slot != nullptr) a.row_of_slot[slot] = row;
          a.prow_of_slot[slot] = prow;
          if (kept) {
            if (a.token_of_row != nullptr) a.token_of_row[row] = t;
            a.slot_of_prow[prow] = (int)slot;
          }
        }
        if (kGates && kept) a.gate_of_prow[prow] = a.gates[slot];
        if (kept && a.tok_of_prow != nullptr) a.tok_of_prow[prow] = t;
        if (kX && kept && a.xs_perm != nullptr) a.xs_perm[prow] = a.xs_tok[t];
      }
      if (!kX && !kDy) continue;   // tables only
      const int ng = min(32, k - jb);
      // kUnroll vectors per lane are loaded before any is stored, so a warp keeps
      // kUnroll x 512 bytes of each source row in flight.  Warp-uniform trip count: every lane
      // takes part in every shuffle, and the vector index is predicated instead (a row need not
      // be a multiple of 32 vectors, e.g. d = 2880).
      for (int v0 = 0; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 vx[kUnroll], vd[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + 32 * u + lane;
          vx[u] = make_uint4(0, 0, 0, 0);
          vd[u] = make_uint4(0, 0, 0, 0);
          if (kX && v < nvec) vx[u] = xs[v];
          if (kDy && v < nvec) vd[u] = dys[v];
        }
        uint2 cx[kUnroll], cd[kUnroll];   // quant: the vectors' codes, stored to every destination
        if constexpr (kQ) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            cx[u] = rx ? encode8_e4m3<true>(vx[u], sx, yx) : encode8_e4m3<false>(vx[u], sx, 0.f);
            cd[u] = rd ? encode8_e4m3<true>(vd[u], sd, yd) : encode8_e4m3<false>(vd[u], sd, 0.f);
          }
        }
        for (int q = 0; q < ng; ++q) {
          const int p = __shfl_sync(0xffffffffu, prow, q);
          if (p < 0) continue;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + 32 * u + lane;
            if (v >= nvec) continue;
            if (kX) reinterpret_cast<uint4*>(a.x_perm + (size_t)p * d)[v] = vx[u];
            if (kDy) reinterpret_cast<uint4*>(a.dy_perm + (size_t)p * d)[v] = vd[u];
            if constexpr (kQ) {
              reinterpret_cast<uint2*>(a.x8 + (size_t)p * d)[v] = cx[u];
              reinterpret_cast<uint2*>(a.dy8 + (size_t)p * d)[v] = cd[u];
            }
          }
          if (kQ && v0 == 0 && lane == 0) {
            a.x8s[p] = sx;
            a.dy8s[p] = sd;
          }
        }
        if (jb == 0) {
          for (int s = 0; s < S; ++s) {
            if (t >= tb->kept[E + s]) continue;
            const size_t p = (size_t)tb->poff[E + s] + t;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
              const int v = v0 + 32 * u + lane;
              if (v >= nvec) continue;
              if (kX) reinterpret_cast<uint4*>(a.x_perm + p * d)[v] = vx[u];
              if (kDy) reinterpret_cast<uint4*>(a.dy_perm + p * d)[v] = vd[u];
              if constexpr (kQ) {
                reinterpret_cast<uint2*>(a.x8 + p * d)[v] = cx[u];
                reinterpret_cast<uint2*>(a.dy8 + p * d)[v] = cd[u];
              }
            }
            if (kQ && v0 == 0 && lane == 0) {
              a.x8s[p] = sx;
              a.dy8s[p] = sd;
            }
          }
        }
      }
    }
    if (lane < S && t < tb->kept[E + lane]) {
      const size_t p = (size_t)tb->poff[E + lane] + t;
      if (kMeta) a.slot_of_prow[p] = -2;
      if (kMeta && a.tok_of_prow != nullptr) a.tok_of_prow[p] = t;
      if (kX && a.xs_perm != nullptr) a.xs_perm[p] = a.xs_tok[t];
      if (kGates) a.gate_of_prow[p] = 1.f;
    }
  }
  // zero the pad rows of every segment
  const int G = tb->G;
  const int total_pad = tb->total_pad;
  for (int p = gw; p < total_pad; p += nw) {
    int lo = 0, hi = G - 1;   // segment g with pad_start[g] <= p < pad_start[g+1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tb->pad_start[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const size_t row = (size_t)tb->poff[lo] + tb->kept[lo] + (p - tb->pad_start[lo]);
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = lane; (kX || kDy) && v < nvec; v += 32) {
      if (kX) reinterpret_cast<uint4*>(a.x_perm + row * d)[v] = z;
      if (kDy) reinterpret_cast<uint4*>(a.dy_perm + row * d)[v] = z;
    }
    if constexpr (kQ) {   // a zero row's codes and scale, as the row quantiser gives them
      for (int v = lane; v < d / 16; v += 32) {
        reinterpret_cast<uint4*>(a.x8 + row * d)[v] = z;
        reinterpret_cast<uint4*>(a.dy8 + row * d)[v] = z;
      }
      if (lane == 0) {
        a.x8s[row] = 1.f;
        a.dy8s[row] = 1.f;
      }
    }
    if (lane == 0) {
      if (kMeta) a.slot_of_prow[row] = -1;
      // a pad row gathers token 0: with a zero gate its dA, dB and Hg are exactly zero
      if (kMeta && a.tok_of_prow != nullptr) a.tok_of_prow[row] = 0;
      if (kX && a.xs_perm != nullptr) a.xs_perm[row] = 0.f;
      if (kGates) a.gate_of_prow[row] = 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_dispatch_scan(const Cfg& c, const Layout& L, const DispatchArgs& a, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(reinterpret_cast<char*>(a.hdr) + kHdrResetOffset, 0, kHdrResetBytes, s);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(a.scan_status, 0, (size_t)L.nscan * c.E * sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  const int N = c.T * c.k;
  prof_mark(kKScan, s, true);
  dispatch_scan_kernel<<<L.nscan, kScanThreads, 0, s>>>(a, N, c.T, c.E, c.S, c.C, L.nscan, L.rows);
  prof_mark(kKScan, s, false);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_gather(const Cfg& c, const Layout& L, const DispatchArgs& a,
                                   bool write_meta, bool gather_x, bool gather_dy, cudaStream_t s, bool gates,
                                   bool quant) {
  (void)L;
  const int blocks = num_sms() * 8;
  prof_mark(kKGather, s, true);
  if (quant && write_meta && gather_x && gather_dy && a.x8 && a.dy8 && a.x8s && a.dy8s)
    dispatch_gather_kernel<true, true, true, false, true><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else if (quant) {
    prof_mark(kKGather, s, false);
    return cudaErrorInvalidValue;
  } else if (write_meta && gather_x && gather_dy)
    dispatch_gather_kernel<true, true, true, false><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else if (write_meta && gather_x)
    dispatch_gather_kernel<true, true, false, false><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else if (write_meta && !gather_x && !gather_dy && gates)
    dispatch_gather_kernel<true, false, false, true><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else if (write_meta && !gather_x && !gather_dy)
    dispatch_gather_kernel<true, false, false, false><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else if (!write_meta && gather_dy && !gather_x)
    dispatch_gather_kernel<false, false, true, false><<<blocks, 256, 0, s>>>(a, c.T, c.k, c.E, c.S, c.d);
  else {
    prof_mark(kKGather, s, false);
    return cudaErrorInvalidValue;
  }
  prof_mark(kKGather, s, false);
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------------------------
// moe_dispatch_noalloc: the same dispatch with its scratch in a fixed, file-scope device array.
// ---------------------------------------------------------------------------------------------
//
// Some callers cannot allocate device memory for a workspace: code that runs inside a memory
// arena owned by a host framework, under a pool that forbids growth at step time, or on a path
// where the implicit synchronisation of cudaMalloc is not allowed.  For them this entry point
// keeps the dispatch's scratch (header, routing tables, look-back status words, per-slot ranks
// and rows, per-row slots) in `g_noalloc_scratch`, which every device that loads the library
// holds until the process exits.  The host side only ever passes the array's device address,
// taken with cudaGetSymbolAddress while the caller's device is current.  There is no workspace
// error word to read back, so the device-side status of each call goes to the caller's optional
// `status` word instead.

namespace moe {
namespace {

constexpr int kNoAllocMaxSlots = 1 << 18;                 // T*k assignments
constexpr int kNoAllocMaxRows = 3 << 17;                  // padded expert-ordered rows
constexpr int kNoAllocMaxScanBlocks = kNoAllocMaxSlots / kScanChunk;

struct NoAllocScratch {
  Hdr hdr;
  Tables tabs;
  uint32_t scan_status[kNoAllocMaxScanBlocks * kMaxE];
  int32_t rank[kNoAllocMaxSlots];
  int32_t prow_of_slot[kNoAllocMaxSlots];
  int32_t slot_of_prow[kNoAllocMaxRows];
};

__device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

// Device address of the scratch array on the current device.  Looked up on every call (a host-side
// table lookup): an address cached per device ordinal would go stale if the caller reset the
// device or released and re-created its primary context, which can reload the module elsewhere.
moe_status_t noalloc_scratch(NoAllocScratch** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  *out = static_cast<NoAllocScratch*>(p);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const int32_t* idx,
                                             const moe_bf16* x, int32_t* counts, int32_t* offsets,
                                             int32_t* row_of_slot, int32_t* token_of_row,
                                             moe_bf16* x_perm, int32_t* status, moe_stream_t stream) {
  using namespace moe;
  Cfg c;
  moe_status_t st = make_cfg(cfg, &c);
  if (st != MOE_OK) return st;
  const void* ptrs[] = {idx, x, counts, offsets, row_of_slot, token_of_row, x_perm};
  for (const void* p : ptrs)
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_ERR_INVALID_ARG;
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(c);
  if ((int64_t)c.T * c.k > kNoAllocMaxSlots || L.rows > kNoAllocMaxRows || L.nscan > kNoAllocMaxScanBlocks)
    return MOE_ERR_UNSUPPORTED;
  if ((st = check_device()) != MOE_OK) return st;
  NoAllocScratch* sc = nullptr;
  if ((st = noalloc_scratch(&sc)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: start from a clean header (error word,
  // look-back counters, test hooks); the scan clears its status words itself.
  if (cudaMemsetAsync(&sc->hdr, 0, sizeof(Hdr), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  DispatchArgs a{};
  a.idx = idx;
  a.x = reinterpret_cast<const uint16_t*>(x);
  a.counts = counts;
  a.offsets = offsets;
  a.row_of_slot = row_of_slot;
  a.token_of_row = token_of_row;
  a.x_perm = reinterpret_cast<uint16_t*>(x_perm);
  a.hdr = &sc->hdr;
  a.tabs = &sc->tabs;
  a.scan_status = sc->scan_status;
  a.rank = sc->rank;
  a.prow_of_slot = sc->prow_of_slot;
  a.slot_of_prow = sc->slot_of_prow;
  a.status_out = status;
  cudaError_t e = launch_dispatch_scan(c, L, a, s);
  if (e == cudaSuccess) e = launch_dispatch_gather(c, L, a, true, true, false, s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
