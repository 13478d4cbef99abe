// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// The pages' point (Piper explainer and technical summary: fine-grained experts turn the FFN into
// many tall-and-skinny GEMMs that use the GPU poorly; MoEBlaze, Methodology item 2: fused expert
// kernels with dispatch, and recompute instead of stored activations) is met here by one
// persistent, warp-specialised kernel per GEMM family over all experts at once:
//
//   warp 0      TMA producer: loads operand tiles into a ring of shared-memory stages
//   warp 1      MMA issuer: one thread issues tcgen05.mma into TMEM accumulators, commits each
//               stage back to the producer and each finished tile to the epilogue
//   warps 2..   epilogue (4 or 8 warps): tcgen05.ld of the accumulator (128 lanes = 128 rows),
//               fused element-wise work, bf16 stores
//
// The six expert GEMMs run on CTA pairs (clusters of two): one 256 x 256 tile per pair, each CTA
// loading its own 128 rows of A and its own 128-row half of B, and the even CTA issuing
// tcgen05.mma.cta_group::2, which feeds both halves of B to both SMs.  Per FLOP this halves the
// shared-memory traffic of B against one CTA doing a 128 x 256 tile, which otherwise saturates the
// SM's shared-memory bandwidth (TMA writes plus tensor-core reads) before the tensor cores.
// Rows are the dispatch's padded expert segments (multiples of 256), so every 256-row pair tile
// belongs to one expert and the per-expert tile scheduler is a table walk done identically by
// the three roles of both CTAs (the MMA thread needs only each tile's K-block count, which it
// derives without the walk).  Every wait is bounded (MOE_ERR_TIMEOUT instead of a hang).
//
// Problems (BK = 64, operands bf16, accumulators fp32; pair tiles M = 256 unless noted):
//   FwdGateUp  H    = silu(X Wg^T) * (X Wu^T)              A=X K-major, B=[Wg;Wu] K-major, N=256
//   FwdDown    O    = H Wd^T                               A=H K-major, B=Wd K-major,      N=256
//   BwdDh      dh'  = dY Wd                                A K-major, B MN-major,      N=256
//   BwdFused   a|b  = X [Wg;Wu]^T (recompute); epilogue: h = silu(a) b, dg += dh'.h, dh = g dh',
//              dA = dh b silu'(a), dB = dh silu(a), Hg = g h                         N=256
//   Wgrad      dWg = dA^T X, dWu = dB^T X, dWd = dY^T Hg   A and B MN-major, K = segment rows
//   DgradX     dX   = dA Wg + dB Wu                        A K-major, B MN-major, K = 2 d_ff
//   RouterDwr  dW_r partials = x^T dl over token splits    A and B MN-major, N = E padded to 64,
//              one CTA, M = 128
//   RouterDx   r    = dl W_r^T (the router's share of dx)  A and B K-major, K = E padded to 64,
//              one CTA, M = 128
//   RouterLogits  l = x W_r with W_r in three bf16 parts; epilogue: softmax, top-k, or the
//              router's dlogits                          A and B K-major, N = E padded to 64
//   FwdGateUp8 H    = silu(sx sg (X8 Wg8^T)) * (sx su (X8 Wu8^T)), e4m3 operands (kind::f8f6f4),
//              K blocks of 128 codes, row / channel scales applied in the epilogue      N=256
//   FwdDown8   O    = sh sd (H8 Wd8^T), e4m3 operands, eight epilogue warps             N=256
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {

// In-kernel SM clock (profiling only): while g_clock_on is set, one thread of every CTA of the GEMM
// kernels (lane 0 of its last warp, not the thread that sets the kernel up) adds its clock64 cycles
// and globaltimer nanoseconds from entry to exit to the kernel's pair of sums, so cycles / ns is the
// mean SM clock over the CTAs' lifetimes -- the clock the kernel actually ran at, which a power cap
// lowers well below what a 50 ms nvidia-smi sample sees.
__device__ int g_clock_on;
__device__ unsigned long long g_clock_acc[kKCount][2];

namespace {

struct ClockSpan {
  unsigned long long c0 = 0, n0 = 0;
  bool on = false;
  __device__ void start() {
    on = g_clock_on != 0;
    if (on) {
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(c0));
      n0 = global_ns();
    }
  }
  __device__ void stop(int id) {
    if (!on) return;
    unsigned long long c1;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c1));
    const unsigned long long n1 = global_ns();
    atomicAdd(&g_clock_acc[id][0], c1 - c0);
    atomicAdd(&g_clock_acc[id][1], n1 - n0);
  }
};

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr uint32_t kTileA = kBM * kBK * 2;   // 16 KB: 128 rows x 64 bf16 (K-major)
constexpr uint32_t kBox = 64 * kBK * 2;      // 8 KB: a 64 x 64 box (MN-major)
constexpr int kPairM = 2 * kBM;              // rows of a CTA-pair tile (kRowTile)
constexpr int kChunkM = 16;                  // pair m-tiles per L2 reuse chunk of a segment
static_assert(kPairM == kRowTile, "segments are padded to the pair tile");

struct Job {
  int seg, m0, n0, kiters, kbase, sub;
  uint32_t idesc;   // instruction descriptor, for problems whose N is a runtime value
};

// Defaults of the per-problem hooks; a policy overrides what it needs.
struct PolicyDefaults {
  // k-iteration before which the MMA waits for the epilogue to release the accumulator
  __device__ static int acc_wait_kit(const Job&) { return 0; }
  // Gathered operand rows (the dispatch gather fused into the operand load; CTA-pair problems): 0
  // none; 1 the K-major A tile's 128 rows come from token order (x or dY) through the token of every
  // padded row; 2 the weight gradient's token-side operand (x or dY, MN-major) takes its 64 K rows per
  // stage the same way, as two 64-column boxes.  Either way a CTA's stage takes 32 tile::gather4
  // copies (four 128-byte lines each) from kGatherWarps warps, and one TMA box for the other operand.
  static constexpr int kGather = 0;
  // Tiles numbered from num_tiles on, zero_tiles() of them, that only the epilogue stores (CTA-pair
  // problems): epilogue_zero of each, by the pair's epilogue warps while they wait for an MMA tile.
  static constexpr bool kZeroTiles = false;
  // TMA bytes that complete one stage at k-iteration kit
  __device__ static uint32_t tx_bytes(const Job&, int, uint32_t stage_bytes) { return stage_bytes; }
  // a stateful policy keeps per-lane epilogue state across the jobs of one CTA (epilogue_s)
  static constexpr bool kStateful = false;
  struct EpiState {};
  static constexpr uint32_t kEpiWarpBytes = 0;   // shared memory per epilogue warp (boxes, scratch)
};

struct SegSmem {
  int G;
  int n_mtiles;
  int poff[kMaxG + 1];
  int16_t seg_order[kMaxG];
};

__device__ __forceinline__ void load_segs(SegSmem& s, const Tables* tb) {
  if (threadIdx.x == 0) {
    s.G = tb->G;
    s.n_mtiles = tb->n_mtiles;
  }
  for (int i = threadIdx.x; i <= kMaxG; i += blockDim.x) {
    s.poff[i] = tb->poff[i];
    if (i < kMaxG) s.seg_order[i] = (int16_t)tb->seg_order[i];
  }
}

// Row-tiled problems: tile t -> (segment, 256-row m-tile, n-tile).  Segments in index order;
// inside a segment, chunks of up to 16 m-tiles x all n-tiles with the m-tile fastest, so the CTA
// pairs working at the same time share one operand panel of each kind in L2.
__device__ __forceinline__ Job row_job(const SegSmem& s, int t, int nt, int bn, int kiters) {
  const int mt_of_t = t / nt;
  int lo = 0, hi = s.G - 1;   // last segment whose first m-tile <= mt_of_t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.poff[mid] / kPairM <= mt_of_t) lo = mid; else hi = mid - 1;
  }
  const int seg = lo;
  const int mstart = s.poff[seg] / kPairM;
  const int mt = (s.poff[seg + 1] - s.poff[seg]) / kPairM;
  const int local = t - mstart * nt;
  const int c = local / (kChunkM * nt);
  const int base = c * kChunkM;
  const int cm = min(kChunkM, mt - base);
  const int r = local - c * kChunkM * nt;
  Job j;
  j.seg = seg;
  j.m0 = s.poff[seg] + (base + r % cm) * kPairM;
  j.n0 = (r / cm) * bn;
  j.kiters = kiters;
  j.kbase = 0;
  j.sub = 0;
  return j;
}

// ---------------------------------------------------------------------------------------------
// Problem policies
// ---------------------------------------------------------------------------------------------

// Hooks of the CTA-pair problems: per CTA a stage holds A (128 x 64) and half of B (128 x 64);
// load() gets the pair's job, this CTA's rank and the even CTA's full barrier (cluster address).
struct PairDefaults : PolicyDefaults {
  static constexpr int kStages = 6;                 // 64-wide K blocks of storage
  static constexpr int kSub = 1;                    // K blocks per pipeline slot (one barrier round)
  static constexpr uint32_t kStageBytes = 2 * kTileA;   // one K block: A 128 x 64 + B half 128 x 64
  static constexpr int kAccCols = 256;
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdesc = idesc_bf16(kPairM, 256, false, false);
  static constexpr uint32_t kEpiWarpBytes = 2 * 2048;   // two TMA-store boxes (kEpiBox)
};

// A stage's gathered operand: 128 lines of 128 bytes (64 bf16) from `dst` within the stage, in the
// 128-byte-swizzled layout a TMA box of 128 rows would leave.  Line L is row tok[L] (kGather 1) or
// tok[L % 64] (kGather 2) of the token-order tensor behind `map` (one-row boxes), from column col0
// (L < 64) or col1.
struct GatherOp {
  const CUtensorMap* map;
  int col0, col1;
  uint32_t dst;
};

// Epilogue output goes through shared memory and TMA stores: each epilogue warp writes a [32 rows x
// 32 bf16] box (its TMEM lane quarter x 32 columns, 2 KB) in the layout of a SWIZZLE_64B tensor map
// -- 16-byte chunk q of row r at r * 64 + ((q ^ ((r >> 1) & 3)) * 16), so each 8-lane phase of a
// chunk write hits distinct banks -- and lane 0 stores the box with one bulk tensor copy that
// writes whole lines.  A thread's direct 16-byte stores would instead touch 32 rows per warp
// instruction, with half-filled sectors, on the same L1 the operand loads pass through.
constexpr uint32_t kEpiBox = 32 * 32 * 2;

__device__ __forceinline__ void stage_box(uint8_t* box, int lane, const uint32_t (&pk)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(box + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// Box i of this warp's epilogue (i counts from 0 within one tile): the box used two stores ago is
// free again once at most one bulk group is still reading.
__device__ __forceinline__ uint8_t* claim_box(uint8_t* ebuf, int i, int lane) {
  if (i >= 2) {
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
  }
  return ebuf + (i & 1) * kEpiBox;
}

// After stage_box(): make the box visible to the TMA and store it at (x, y) [, z].
__device__ __forceinline__ void store_box_2d(const CUtensorMap* map, const uint8_t* box, int lane, int x, int y) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, box, x, y);
    bulk_commit();
  }
}

__device__ __forceinline__ void store_box_3d(const CUtensorMap* map, const uint8_t* box, int lane, int x, int y,
                                             int z) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(map, box, x, y, z);
    bulk_commit();
  }
}

// Start of a tile's epilogue: every box of the previous tile has been read.
__device__ __forceinline__ void epi_begin(int lane) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
}

__device__ __forceinline__ void pack32(const uint32_t (&v)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
}

// K-major A and B: kk-th K=16 step of a 64-wide block
__device__ __forceinline__ void mma_kk_kmajor(uint32_t sa, uint32_t dt, uint32_t idesc, int kit) {
#pragma unroll
  for (int kk = 0; kk < kBK / 16; ++kk)
    umma_bf16_pair(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kTileA + kk * 32), idesc, (kit | kk) != 0);
}

// K-major A, MN-major B (two 64-wide boxes)
__device__ __forceinline__ void mma_kk_bmn(uint32_t sa, uint32_t dt, uint32_t idesc, int kit) {
#pragma unroll
  for (int kk = 0; kk < kBK / 16; ++kk)
    umma_bf16_pair(dt, sdesc_kmajor(sa + kk * 32), sdesc_mnmajor(sa + kTileA + kk * 2048, kBox), idesc,
                   (kit | kk) != 0);
}

// H = silu(X Wg^T) * (X Wu^T).  B = [Wg rows n0..n0+127; Wu rows n0..n0+127]: the even CTA loads
// the Wg half and the odd CTA the Wu half, so TMEM columns 0-127 hold the gate and 128-255 the up
// projection of the same 128 hidden units.  kKeep: pair tiles below keep_rows also store a and b
// (bf16) for the backward, from triplets of staging boxes (H, a, b; two triplets per warp, five
// pipeline stages to make room).
template <bool kKeep, bool kG = false>
struct FwdGateUpT : PairDefaults {
  static constexpr int kId = kKGateUp;
  static constexpr int kEpiWarps = 4;
  static constexpr int kStages = kKeep ? 5 : 6;
  static constexpr uint32_t kEpiWarpBytes = kKeep ? 6 * 2048 : 2 * 2048;
  static constexpr int kGather = kG ? 1 : 0;
  struct Params {
    CUtensorMap tmX, tmWg, tmWu, tmH, tmA, tmB;   // tmX: x_perm, or x in token order (gathered)
    const int32_t* tok;                           // gathered: token of every padded row
    int f, d, nt, keep_rows;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 128, p.d / kBK);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return p.d / kBK; }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmX); tma_prefetch(&p.tmWg); tma_prefetch(&p.tmWu);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    if constexpr (!kG) tma_load_2d_pair(st, &p.tmX, cbar, kit * kBK, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, rank ? &p.tmWu : &p.tmWg, cbar, kit * kBK, j.n0, j.seg);
  }
  // gathered: this CTA's 128 rows of the tile, K block kit
  __device__ static const int32_t* gather_tok(const Params& p, const Job& j, int, int rank) {
    return p.tok + j.m0 + kBM * rank;
  }
  __device__ static GatherOp gather_op(const Params& p, const Job&, int kit, int) {
    return GatherOp{&p.tmX, kit * kBK, kit * kBK, 0u};
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
    mma_kk_kmajor(sa, dt, kIdesc, kit);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    const int lane = row & 31;
    const int y = j.m0 + (row & ~31);
    const bool keep = kKeep && y < p.keep_rows;   // whole pair tiles: keep_rows is a multiple of 256
    epi_begin(lane);
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      if (j.n0 + c >= p.f) break;
      uint32_t ga[32], ub[32];
      tmem_ld32(ta + c, ga);
      tmem_ld32(ta + 128 + c, ub);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a0 = __uint_as_float(ga[2 * i]), a1 = __uint_as_float(ga[2 * i + 1]);
        const float h0 = a0 * sigmoid_fast(a0) * __uint_as_float(ub[2 * i]);
        const float h1 = a1 * sigmoid_fast(a1) * __uint_as_float(ub[2 * i + 1]);
        pk[i] = pack_bf16(h0, h1);
      }
      if (!kKeep) {
        uint8_t* box = claim_box(ebuf, c / 32, lane);
        stage_box(box, lane, pk);
        store_box_2d(&p.tmH, box, lane, j.n0 + c, y);
        continue;
      }
      const int i = c / 32;
      if (i >= 2) {   // the triplet used two pieces ago has been read
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
      }
      uint8_t* box = ebuf + (i & 1) * 3 * kEpiBox;
      stage_box(box, lane, pk);
      if (keep) {
        uint32_t pa[16], pb[16];
        pack32(ga, pa);
        pack32(ub, pb);
        stage_box(box + kEpiBox, lane, pa);
        stage_box(box + 2 * kEpiBox, lane, pb);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmH, box, j.n0 + c, y);
        if (keep) {
          tma_store_2d(&p.tmA, box + kEpiBox, j.n0 + c, y);
          tma_store_2d(&p.tmB, box + 2 * kEpiBox, j.n0 + c, y);
        }
        bulk_commit();
      }
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};
using FwdGateUp = FwdGateUpT<false>;
using FwdGateUpG = FwdGateUpT<false, true>;

// The gate/up projection with FP8 operands (tcgen05 kind::f8f6f4, e4m3): x_perm rows and W_gate /
// W_up rows quantised per row (codes and an fp32 scale each), so a = s_x s_g (q_x . q_g) exactly
// up to the fp32 accumulation.  Same pair tiling as FwdGateUp: a K block is 128 e4m3 values (the
// same 128 bytes per row as 64 bf16), four K = 32 MMAs per block; the epilogue applies the row
// scale and the output channel's scale before SwiGLU.
struct FwdGateUp8 : PairDefaults {
  static constexpr int kId = kKGateUpFp8;
  static constexpr int kEpiWarps = 4;
  static constexpr int kBK8 = 128;
  static constexpr uint32_t kIdesc = idesc_e4m3(kPairM, 256);
  struct Params {
    CUtensorMap tmX, tmWg, tmWu, tmH;
    const float *xs, *gs, *us;   // [rows] and [G, f] scales
    int f, d, nt;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 128, (p.d + kBK8 - 1) / kBK8);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return (p.d + kBK8 - 1) / kBK8; }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmX); tma_prefetch(&p.tmWg); tma_prefetch(&p.tmWu);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    tma_load_2d_pair(st, &p.tmX, cbar, kit * kBK8, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, rank ? &p.tmWu : &p.tmWg, cbar, kit * kBK8, j.n0, j.seg);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_f8_pair(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kTileA + kk * 32), kIdesc, (kit | kk) != 0);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    const int lane = row & 31;
    const int y = j.m0 + (row & ~31);
    const float sx = p.xs[j.m0 + row];
    const float* gs = p.gs + (size_t)j.seg * p.f + j.n0;
    const float* us = p.us + (size_t)j.seg * p.f + j.n0;
    epi_begin(lane);
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
      if (j.n0 + c >= p.f) break;
      uint32_t ga[32], ub[32];
      tmem_ld32(ta + c, ga);
      tmem_ld32(ta + 128 + c, ub);
      tmem_ld_wait();
      float sg[32], su[32];   // the 32 columns' weight scales (the same for every lane)
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(gs + c) + v);
        const float4 u4 = __ldg(reinterpret_cast<const float4*>(us + c) + v);
        sg[4 * v] = g4.x; sg[4 * v + 1] = g4.y; sg[4 * v + 2] = g4.z; sg[4 * v + 3] = g4.w;
        su[4 * v] = u4.x; su[4 * v + 1] = u4.y; su[4 * v + 2] = u4.z; su[4 * v + 3] = u4.w;
      }
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float hv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float a = __uint_as_float(ga[2 * i + h]) * sx * sg[2 * i + h];
          hv[h] = a * sigmoid_fast(a) * (__uint_as_float(ub[2 * i + h]) * sx * su[2 * i + h]);
        }
        pk[i] = pack_bf16(hv[0], hv[1]);
      }
      uint8_t* box = claim_box(ebuf, c / 32, lane);
      stage_box(box, lane, pk);
      store_box_2d(&p.tmH, box, lane, j.n0 + c, y);
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// Out = (s_a A8)(s_b B8[g])^T with e4m3 operands, both K-major: A [rows, K] codes with one scale
// per row, B[g] [N, K] codes with one scale per output channel; N = 256 columns per pair tile, each
// CTA loading 128 rows of B[g]; 128-wide K blocks (the last one zero-filled past K).  The epilogue
// scales the fp32 accumulator by s_a[row] s_b[g, col] and stores bf16.  Three problems have this
// shape (one kernel each, by kId_):
//   FwdDown8   O   = H8 Wd8^T         A = h rows (K = d_ff),       B = W_down rows (N = d_model)
//   BwdDh8     dh' = dY8 WdT8^T       A = dY rows (K = d_model),   B = W_down's columns (N = d_ff)
//   DgradX8    dX  = dAB8 WguT8^T     A = [dA | dB] rows (K = 2 d_ff), B = column i of W_gate and W_up
//                                     together (N = d_model)
template <int kId_>
struct RowChan8 : PairDefaults {
  static constexpr int kId = kId_;
  // two epilogue warps per TMEM lane quarter, 128 columns each: with K blocks twice as deep as
  // bf16's, a short K (6 to 11 blocks) leaves the main loop shorter than one warp's 256 columns
  static constexpr int kEpiWarps = 8;
  static constexpr int kBK8 = 128;
  static constexpr uint32_t kIdesc = idesc_e4m3(kPairM, 256);
  struct Params {
    CUtensorMap tmA, tmB, tmO;
    const float *as, *bs;   // [rows] and [G, N] scales
    int K, N, nt;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 256, (p.K + kBK8 - 1) / kBK8);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return (p.K + kBK8 - 1) / kBK8; }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmA); tma_prefetch(&p.tmB); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    tma_load_2d_pair(st, &p.tmA, cbar, kit * kBK8, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, &p.tmB, cbar, kit * kBK8, j.n0 + kBM * rank, j.seg);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_f8_pair(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kTileA + kk * 32), kIdesc, (kit | kk) != 0);
  }
  // Two 32-column boxes per round: both TMEM loads and the 64 column scales are in flight together,
  // and one proxy fence covers both boxes' stores.
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int part, int,
                                  uint8_t* ebuf) {
    const int lane = row & 31;
    const int y = j.m0 + (row & ~31);
    const float sh = p.as[j.m0 + row];
    const float* ds = p.bs + (size_t)j.seg * p.N + j.n0;
    epi_begin(lane);
#pragma unroll 1
    for (int c = part * 128; c < part * 128 + 128; c += 64) {
      if (j.n0 + c >= p.N) break;   // N is a multiple of 64: a round's two boxes both exist
      uint32_t v[2][32];
      tmem_ld32(ta + c, v[0]);
      tmem_ld32(ta + c + 32, v[1]);
      float4 s4[16];                // the 64 columns' weight scales (the same for every lane)
#pragma unroll
      for (int q = 0; q < 16; ++q) s4[q] = __ldg(reinterpret_cast<const float4*>(ds + c) + q);
      tmem_ld_wait();
      if (c != part * 128) {        // the previous round's boxes have been read by their stores
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
#pragma unroll
      for (int bx = 0; bx < 2; ++bx) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 sc = s4[bx * 8 + i / 2];
          const float s0 = (i & 1) ? sc.z : sc.x, s1 = (i & 1) ? sc.w : sc.y;
          pk[i] = pack_bf16(__uint_as_float(v[bx][2 * i]) * sh * s0, __uint_as_float(v[bx][2 * i + 1]) * sh * s1);
        }
        stage_box(ebuf + bx * kEpiBox, lane, pk);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmO, ebuf, j.n0 + c, y);
        tma_store_2d(&p.tmO, ebuf + kEpiBox, j.n0 + c + 32, y);
        bulk_commit();
      }
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};
using FwdDown8 = RowChan8<kKDownFp8>;
using BwdDh8 = RowChan8<kKBwdDhFp8>;
using DgradX8 = RowChan8<kKDgradXFp8>;

// Shared by FwdDown, BwdDh and DgradX: this warp's 32 rows of the fp32 accumulator [128 x 256] ->
// bf16 boxes of the output [rows, ncols] at row y (the warp's first row) and columns n0 + c.
__device__ __forceinline__ void store_acc_boxes(const CUtensorMap* map, int y, int n0, int ncols, uint32_t ta,
                                                int lane, uint8_t* ebuf, int cbeg = 0, int cend = 256) {
  epi_begin(lane);
#pragma unroll 1
  for (int c = cbeg; c < cend; c += 32) {
    if (n0 + c >= ncols) break;
    uint32_t v[32];
    tmem_ld32(ta + c, v);
    tmem_ld_wait();
    uint32_t pk[16];
    pack32(v, pk);
    uint8_t* box = claim_box(ebuf, (c - cbeg) / 32, lane);
    stage_box(box, lane, pk);
    store_box_2d(map, box, lane, n0 + c, y);
  }
}

// O = H Wd^T: N = 256 columns of d_model, each CTA loading 128 rows of Wd[e].
struct FwdDown : PairDefaults {
  static constexpr int kId = kKDown;
  static constexpr int kEpiWarps = 4;
  struct Params {
    CUtensorMap tmH, tmWd, tmO;
    int f, d, nt;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 256, p.f / kBK);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return p.f / kBK; }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmH); tma_prefetch(&p.tmWd); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    tma_load_2d_pair(st, &p.tmH, cbar, kit * kBK, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, &p.tmWd, cbar, kit * kBK, j.n0 + kBM * rank, j.seg);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
    mma_kk_kmajor(sa, dt, kIdesc, kit);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    store_acc_boxes(&p.tmO, j.m0 + (row & ~31), j.n0, p.d, ta, row & 31, ebuf);
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// dh' = dY W_d for every row tile: N = 256 columns of d_ff, K = d_model.  W_d[e] is
// [d_model, d_ff], so it is the MN-major B operand (two 64-wide boxes per CTA and stage).  dh' is
// stored in bf16 for the SwiGLU backward below.
template <bool kG>
struct BwdDhT : PairDefaults {
  static constexpr int kId = kKBwdDh;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kIdesc = idesc_bf16(kPairM, 256, false, true);
  static constexpr int kGather = kG ? 1 : 0;
  struct Params {
    CUtensorMap tmDY, tmWdT, tmDH;   // tmDY: dY_perm, or dy in token order (gathered)
    const int32_t* tok;              // gathered: token of every padded row
    int f, d, nt;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 256, p.d / kBK);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return p.d / kBK; }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmDY); tma_prefetch(&p.tmWdT); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    if constexpr (!kG) tma_load_2d_pair(st, &p.tmDY, cbar, kit * kBK, j.m0 + kBM * rank);
    tma_load_4d_pair(st + kTileA, &p.tmWdT, cbar, 0, kit * kBK, (j.n0 + kBM * rank) / 64, j.seg);
  }
  // gathered: this CTA's 128 rows of the tile, K block kit
  __device__ static const int32_t* gather_tok(const Params& p, const Job& j, int, int rank) {
    return p.tok + j.m0 + kBM * rank;
  }
  __device__ static GatherOp gather_op(const Params& p, const Job&, int kit, int) {
    return GatherOp{&p.tmDY, kit * kBK, kit * kBK, 0u};
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
    mma_kk_bmn(sa, dt, kIdesc, kit);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    store_acc_boxes(&p.tmDH, j.m0 + (row & ~31), j.n0, p.f, ta, row & 31, ebuf);
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};
using BwdDh = BwdDhT<false>;
using BwdDhG = BwdDhT<true>;

// The recompute a | b = X [Wg;Wu]^T (the forward's first GEMM shape, double-buffered TMEM) with the
// SwiGLU backward in its epilogue, which reads this tile's dh' written by BwdDh:
//   h = silu(a) b, dg += dh'.h, dh = g dh', dA = dh b silu'(a), dB = dh silu(a), Hg = g h.
// Four epilogue warps, one per TMEM lane quarter (eight, two per quarter, measured 77% instead of
// 84% of the MMA rate per SM cycle).  dg is summed per 64-column half of the tile.
template <bool kG>
struct BwdFusedT : PairDefaults {
  static constexpr int kId = kKBwdFused;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kEpiWarpBytes = 3 * 2048;   // boxes for dA, dB, Hg
  static constexpr int kGather = kG ? 1 : 0;
  struct Params {
    CUtensorMap tmX, tmWg, tmWu, tmDA, tmDB, tmHg;   // tmX: x_perm, or x in token order (gathered)
    const int32_t* tok;                              // gathered: token of every padded row
    const uint16_t* DH;
    const float* gate_of_prow;
    float* dg_part;
    int f, d, nt, ndg, keep_rows;   // pair tiles below keep_rows come from the kept a, b instead
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    Job j = row_job(s, t, p.nt, 128, p.d / kBK);
    if (j.m0 < p.keep_rows) j.kiters = 0;
    return j;
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { return p.keep_rows > 0 ? job(p, s, t).kiters : p.d / kBK; }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmX); tma_prefetch(&p.tmWg); tma_prefetch(&p.tmWu);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    if constexpr (!kG) tma_load_2d_pair(st, &p.tmX, cbar, kit * kBK, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, rank ? &p.tmWu : &p.tmWg, cbar, kit * kBK, j.n0, j.seg);
  }
  // gathered: this CTA's 128 rows of the tile, K block kit
  __device__ static const int32_t* gather_tok(const Params& p, const Job& j, int, int rank) {
    return p.tok + j.m0 + kBM * rank;
  }
  __device__ static GatherOp gather_op(const Params& p, const Job&, int kit, int) {
    return GatherOp{&p.tmX, kit * kBK, kit * kBK, 0u};
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
    mma_kk_kmajor(sa, dt, kIdesc, kit);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int part, int,
                                  uint8_t* ebuf) {
    const int lane = row & 31;
    const int y = j.m0 + (row & ~31);
    const size_t r = (size_t)(j.m0 + row);
    const float g = p.gate_of_prow[r];
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float dg = 0.f;
  #pragma unroll 1
      for (int c = half * 64; c < half * 64 + 64; c += 32) {
        if (j.n0 + c >= p.f) break;
        const uint4* dsrc = reinterpret_cast<const uint4*>(p.DH + r * p.f + j.n0 + c);
        uint4 dv[4];
  #pragma unroll
        for (int q = 0; q < 4; ++q) dv[q] = dsrc[q];
        uint32_t va[32], vb[32];
        tmem_ld32(ta + c, va);
        tmem_ld32(ta + 128 + c, vb);
        tmem_ld_wait();
        const uint32_t du[16] = {dv[0].x, dv[0].y, dv[0].z, dv[0].w, dv[1].x, dv[1].y, dv[1].z, dv[1].w,
                                 dv[2].x, dv[2].y, dv[2].z, dv[2].w, dv[3].x, dv[3].y, dv[3].z, dv[3].w};
        uint32_t pa[16], pb[16], ph[16];
  #pragma unroll
        for (int i = 0; i < 16; ++i) {
          float o_da[2], o_db[2], o_h[2];
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float a = __uint_as_float(va[2 * i + h]);
            const float b = __uint_as_float(vb[2 * i + h]);
            const float dhp = h ? bf16_hi(du[i]) : bf16_lo(du[i]);
            const float sg = sigmoid_fast(a);
            const float sa = a * sg;
            const float hv = sa * b;
            dg = fmaf(dhp, hv, dg);
            const float dh = g * dhp;
            o_da[h] = dh * b * sg * (1.f + a * (1.f - sg));
            o_db[h] = dh * sa;
            o_h[h] = g * hv;
          }
          pa[i] = pack_bf16(o_da[0], o_da[1]);
          pb[i] = pack_bf16(o_db[0], o_db[1]);
          ph[i] = pack_bf16(o_h[0], o_h[1]);
        }
        if (lane == 0) bulk_wait_read<0>();   // the previous boxes have been read
        __syncwarp();
        stage_box(ebuf, lane, pa);
        stage_box(ebuf + kEpiBox, lane, pb);
        stage_box(ebuf + 2 * kEpiBox, lane, ph);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tmDA, ebuf, j.n0 + c, y);
          tma_store_2d(&p.tmDB, ebuf + kEpiBox, j.n0 + c, y);
          tma_store_2d(&p.tmHg, ebuf + 2 * kEpiBox, j.n0 + c, y);
          bulk_commit();
        }
      }
      p.dg_part[r * p.ndg + (j.n0 / 128) * 2 + half] = dg;
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};
using BwdFused = BwdFusedT<false>;
using BwdFusedG = BwdFusedT<true>;

// The FP8 backward's recompute: a | b = s_x s_g (X8 Wg8^T) | s_x s_u (X8 Wu8^T) from the forward's
// e4m3 codes (FwdGateUp8's main loop), with BwdFused's SwiGLU backward in the epilogue reading this
// tile's dh' (written by BwdDh8):
//   h = silu(a) b, dg += dh'.h, dh = g dh', dA = dh b silu'(a), dB = dh silu(a), Hg = g h.
struct BwdFused8 : PairDefaults {
  static constexpr int kId = kKBwdFusedFp8;
  static constexpr int kEpiWarps = 4;
  static constexpr int kBK8 = 128;
  static constexpr uint32_t kIdesc = idesc_e4m3(kPairM, 256);
  static constexpr uint32_t kEpiWarpBytes = 3 * 2048;   // boxes for dA, dB, Hg
  struct Params {
    CUtensorMap tmX, tmWg, tmWu, tmDA, tmDB, tmHg;
    const float *xs, *gs, *us;   // [rows] and [G, f] scales
    const uint16_t* DH;
    const float* gate_of_prow;
    float* dg_part;
    int f, d, nt, ndg;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 128, (p.d + kBK8 - 1) / kBK8);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return (p.d + kBK8 - 1) / kBK8; }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmX); tma_prefetch(&p.tmWg); tma_prefetch(&p.tmWu);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    tma_load_2d_pair(st, &p.tmX, cbar, kit * kBK8, j.m0 + kBM * rank);
    tma_load_3d_pair(st + kTileA, rank ? &p.tmWu : &p.tmWg, cbar, kit * kBK8, j.n0, j.seg);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_f8_pair(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kTileA + kk * 32), kIdesc, (kit | kk) != 0);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    const int lane = row & 31;
    const int y = j.m0 + (row & ~31);
    const size_t r = (size_t)(j.m0 + row);
    const float g = p.gate_of_prow[r];
    const float sx = p.xs[r];
    const float* gsp = p.gs + (size_t)j.seg * p.f + j.n0;
    const float* usp = p.us + (size_t)j.seg * p.f + j.n0;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      float dg = 0.f;
#pragma unroll 1
      for (int c = half * 64; c < half * 64 + 64; c += 32) {
        if (j.n0 + c >= p.f) break;
        const uint4* dsrc = reinterpret_cast<const uint4*>(p.DH + r * p.f + j.n0 + c);
        uint4 dv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) dv[q] = dsrc[q];
        uint32_t va[32], vb[32];
        tmem_ld32(ta + c, va);
        tmem_ld32(ta + 128 + c, vb);
        float sg[32], su[32];   // the 32 columns' weight scales (the same for every lane)
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 g4 = __ldg(reinterpret_cast<const float4*>(gsp + c) + v);
          const float4 u4 = __ldg(reinterpret_cast<const float4*>(usp + c) + v);
          sg[4 * v] = g4.x; sg[4 * v + 1] = g4.y; sg[4 * v + 2] = g4.z; sg[4 * v + 3] = g4.w;
          su[4 * v] = u4.x; su[4 * v + 1] = u4.y; su[4 * v + 2] = u4.z; su[4 * v + 3] = u4.w;
        }
        tmem_ld_wait();
        const uint32_t du[16] = {dv[0].x, dv[0].y, dv[0].z, dv[0].w, dv[1].x, dv[1].y, dv[1].z, dv[1].w,
                                 dv[2].x, dv[2].y, dv[2].z, dv[2].w, dv[3].x, dv[3].y, dv[3].z, dv[3].w};
        uint32_t pa[16], pb[16], ph[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float o_da[2], o_db[2], o_h[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float a = __uint_as_float(va[2 * i + h]) * sx * sg[2 * i + h];
            const float b = __uint_as_float(vb[2 * i + h]) * sx * su[2 * i + h];
            const float dhp = h ? bf16_hi(du[i]) : bf16_lo(du[i]);
            const float sgm = sigmoid_fast(a);
            const float sa = a * sgm;
            const float hv = sa * b;
            dg = fmaf(dhp, hv, dg);
            const float dh = g * dhp;
            o_da[h] = dh * b * sgm * (1.f + a * (1.f - sgm));
            o_db[h] = dh * sa;
            o_h[h] = g * hv;
          }
          pa[i] = pack_bf16(o_da[0], o_da[1]);
          pb[i] = pack_bf16(o_db[0], o_db[1]);
          ph[i] = pack_bf16(o_h[0], o_h[1]);
        }
        if (lane == 0) bulk_wait_read<0>();   // the previous boxes have been read
        __syncwarp();
        stage_box(ebuf, lane, pa);
        stage_box(ebuf + kEpiBox, lane, pb);
        stage_box(ebuf + 2 * kEpiBox, lane, ph);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tmDA, ebuf, j.n0 + c, y);
          tma_store_2d(&p.tmDB, ebuf + kEpiBox, j.n0 + c, y);
          tma_store_2d(&p.tmHg, ebuf + 2 * kEpiBox, j.n0 + c, y);
          bulk_commit();
        }
      }
      p.dg_part[r * p.ndg + (j.n0 / 128) * 2 + half] = dg;
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// dX = dA Wg + dB Wu: K = 2 d_ff (the dA blocks, then the dB blocks), N = 256 columns of d_model;
// Wg[e], Wu[e] are [d_ff, d_model], so B is MN-major (two 64-wide boxes per CTA and stage).
struct DgradX : PairDefaults {
  static constexpr int kId = kKDgradX;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kIdesc = idesc_bf16(kPairM, 256, false, true);
  struct Params {
    CUtensorMap tmDA, tmDB, tmWgT, tmWuT, tmDX;
    int f, d, nt;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return s.n_mtiles * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    return row_job(s, t, p.nt, 256, 2 * p.f / kBK);
  }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) { (void)s; (void)t; return 2 * p.f / kBK; }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmDA); tma_prefetch(&p.tmDB); tma_prefetch(&p.tmWgT); tma_prefetch(&p.tmWuT);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    const int nk = p.f / kBK;
    const bool up = kit >= nk;
    const int k0 = (up ? kit - nk : kit) * kBK;
    tma_load_2d_pair(st, up ? &p.tmDB : &p.tmDA, cbar, k0, j.m0 + kBM * rank);
    tma_load_4d_pair(st + kTileA, up ? &p.tmWuT : &p.tmWgT, cbar, 0, k0, (j.n0 + kBM * rank) / 64, j.seg);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
    mma_kk_bmn(sa, dt, kIdesc, kit);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int, uint8_t* ebuf) {
    store_acc_boxes(&p.tmDX, j.m0 + (row & ~31), j.n0, p.d, ta, row & 31, ebuf);
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// Weight gradients, K = the expert's rows: dWg = dA^T X and dWu = dB^T X (M = d_ff, N = d_model),
// dWd = dY^T Hg (M = d_model, N = d_ff).  A and B are row-major activations read MN-major: two
// 64 x 64 boxes each per CTA and stage, fetched by one copy (map_mn2; two copies per operand held
// the kernel at 73% of the MMA rate per SM cycle, one copy reaches 86%).  Tiles go expert by
// expert, largest first (experts with no rows spread among them, tile_of); inside an expert the
// d_model-wide operand (X, or dY) is the one cycled through, so the pairs at work keep all of it
// and a few d_ff-wide column blocks in L2.
template <bool kG>
struct WgradT : PairDefaults {
  static constexpr int kId = kKWgrad;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kIdesc = idesc_bf16(kPairM, 256, true, true);
  static constexpr int kGather = kG ? 2 : 0;
  static constexpr bool kZeroTiles = true;
  struct Params {
    CUtensorMap tmDA, tmDB, tmX, tmDY, tmHg;   // all [rows, width] as 64-column block pairs (map_mn2);
                                               // gathered: tmX, tmDY are x, dy in token order, one-row boxes
    CUtensorMap tmdWg, tmdWu, tmdWd;           // [G, M, ncols] with 32 x 32 boxes (stores)
    const int32_t* tok;                        // gathered: token of every padded row
    uint16_t *dWg, *dWu, *dWd;
    int f, d;
    int mt_f, nt_d, mt_d, nt_f, tps;           // pair tiles: dWg/dWu (mt_f x nt_d), dWd (mt_d x nt_f)
    Hdr* hdr;
    const Tables* tabs;
  };
  // The MMA tiles are those of experts with rows, largest first (seg_order).  The tiles of experts
  // with none -- a zero gradient each, no MMA -- come after them in the same numbering; the
  // epilogue warps store them in between their MMA tiles (zero_tiles).
  __device__ static int nonempty(const SegSmem& s) {
    int lo = 0, hi = s.G;   // first position of seg_order whose segment is empty
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      const int g = s.seg_order[mid];
      if (s.poff[g + 1] > s.poff[g]) lo = mid + 1; else hi = mid;
    }
    return lo;
  }
  __device__ static int num_tiles(const Params& p, const SegSmem& s) { return nonempty(s) * p.tps; }
  __device__ static int zero_tiles(const Params& p, const SegSmem& s) { return (s.G - nonempty(s)) * p.tps; }
  __device__ static int mma_kiters(const Params& p, const SegSmem& s, int t) {
    const int g = s.seg_order[t / p.tps];
    return (s.poff[g + 1] - s.poff[g]) / kBK;
  }
  __device__ static Job job(const Params& p, const SegSmem& s, int t) {
    const int pos = t / p.tps;
    int r = t - pos * p.tps;
    Job j;
    j.seg = s.seg_order[pos];
    j.kbase = s.poff[j.seg];
    j.kiters = (s.poff[j.seg + 1] - s.poff[j.seg]) / kBK;
    const int gu = p.mt_f * p.nt_d;
    if (r < 2 * gu) {
      j.sub = r / gu;
      r -= j.sub * gu;
      j.m0 = (r / p.nt_d) * kPairM;
      j.n0 = (r % p.nt_d) * 256;
    } else {   // dWd: m fastest, so the pairs at work share a few Hg column blocks (d_ff wide)
      r -= 2 * gu;
      j.sub = 2;
      j.m0 = (r % p.mt_d) * kPairM;
      j.n0 = (r / p.mt_d) * 256;
    }
    return j;
  }
  __device__ static void prefetch(const Params& p) {
    tma_prefetch(&p.tmDA); tma_prefetch(&p.tmDB); tma_prefetch(&p.tmX); tma_prefetch(&p.tmDY);
    tma_prefetch(&p.tmHg);
  }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint32_t cbar, int rank) {
    const int row = j.kbase + kit * kBK;
    if constexpr (kG) {   // the operand of the other side only; the token-side one is gathered
      if (j.sub == 2) tma_load_3d_pair(st + 2 * kBox, &p.tmHg, cbar, 0, row, (j.n0 + kBM * rank) / 64);
      else tma_load_3d_pair(st, j.sub == 0 ? &p.tmDA : &p.tmDB, cbar, 0, row, (j.m0 + kBM * rank) / 64);
      return;
    }
    const CUtensorMap* ta = j.sub == 0 ? &p.tmDA : (j.sub == 1 ? &p.tmDB : &p.tmDY);
    const CUtensorMap* tb = j.sub == 2 ? &p.tmHg : &p.tmX;
    tma_load_3d_pair(st, ta, cbar, 0, row, (j.m0 + kBM * rank) / 64);
    tma_load_3d_pair(st + 2 * kBox, tb, cbar, 0, row, (j.n0 + kBM * rank) / 64);
  }
  // The token-side operand, MN-major: its 64 K rows (this stage's padded rows) x this CTA's 128
  // columns, as two 64-column boxes (dY for dWd in the A place, x for dWg / dWu in the B place).  A
  // column block past d_model (the last tile of a width not a multiple of 256) is clamped onto the
  // last block: those accumulator rows or columns are never stored.
  __device__ static const int32_t* gather_tok(const Params& p, const Job& j, int kit, int) {
    return p.tok + j.kbase + kit * kBK;
  }
  __device__ static GatherOp gather_op(const Params& p, const Job& j, int, int rank) {
    const int c = (j.sub == 2 ? j.m0 : j.n0) + kBM * rank;
    return GatherOp{j.sub == 2 ? &p.tmDY : &p.tmX, min(c, p.d - 64), min(c + 64, p.d - 64),
                    j.sub == 2 ? 0u : 2 * kBox};
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)
      umma_bf16_pair(dt, sdesc_mnmajor(sa + kk * 2048, kBox), sdesc_mnmajor(sa + 2 * kBox + kk * 2048, kBox),
                     kIdesc, (kit | kk) != 0);
  }
  // Four epilogue warps, one per TMEM lane quarter, 256 columns each (eight warps sharing the
  // quarters measured 3% fewer MMA cycles per SM cycle).  A warp whose 32 rows all lie past M
  // (the last pair tile of a d_ff or d_model not a multiple of 256) stores nothing; boxes that
  // reach past M are clipped by the tensor map.
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int part, int,
                                  uint8_t* ebuf) {
    const int lane = row & 31;
    const int M = j.sub == 2 ? p.d : p.f;
    const int ncols = j.sub == 2 ? p.f : p.d;
    const int y = j.m0 + (row & ~31);
    if (y >= M) return;
    const CUtensorMap* map = j.sub == 0 ? &p.tmdWg : (j.sub == 1 ? &p.tmdWu : &p.tmdWd);
    epi_begin(lane);
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      if (j.n0 + c >= ncols) break;
      uint32_t v[32];
      tmem_ld32(ta + c, v);
      tmem_ld_wait();
      uint32_t pk[16];
      pack32(v, pk);
      uint8_t* box = claim_box(ebuf, c / 32, lane);
      stage_box(box, lane, pk);
      store_box_3d(map, box, lane, j.n0 + c, y, j.seg);
    }
  }
  // An expert that received no rows has a zero gradient.  The warp stores its 32 rows of the tile
  // one row at a time, 16 bytes a lane: 256 columns, whole lines per instruction.
  __device__ static void epilogue_zero(const Params& p, const Job& j, int row, int) {
    const int lane = row & 31;
    const int M = j.sub == 2 ? p.d : p.f;
    const int ncols = j.sub == 2 ? p.f : p.d;
    uint16_t* W = j.sub == 0 ? p.dWg : (j.sub == 1 ? p.dWu : p.dWd);
    const int c = j.n0 + 8 * lane;
    for (int i = 0; i < 32; ++i) {
      const int m = j.m0 + (row & ~31) + i;
      if (m >= M) break;
      if (c < ncols) *reinterpret_cast<uint4*>(W + ((size_t)j.seg * M + m) * ncols + c) = make_uint4(0, 0, 0, 0);
    }
  }
};
using Wgrad = WgradT<false>;
using WgradG = WgradT<true>;

// Router weight gradient on the tensor cores: partial[split][i][e] = sum over the split's tokens of
// x[t][i] dl[t][e].  M = d_model in 128-row tiles (A = x, MN-major), N = E padded to 64 (B = the
// bf16 dlogits [T, Ep], MN-major, NB = Ep / 64 boxes), K = the split's tokens (tensor maps zero-fill
// past T).  The product is one read of x, so the stages are sized by NB: as many as fit, to keep
// x in flight.  The splits are summed in a fixed order afterwards, so the result is deterministic.
template <int NB>
struct RouterDwrT : PolicyDefaults {
  static constexpr int kId = kKRouterDwr;
  static constexpr int kEpiWarps = 4;
  static constexpr uint32_t kStageBytes = (2 + NB) * kBox;
  static constexpr int kStages = (int)(196u * 1024u / kStageBytes) < 8 ? (int)(196u * 1024u / kStageBytes) : 8;
  static constexpr int kAccCols = 256;
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = 512;
  struct Params {
    CUtensorMap tmX, tmDL;
    float* part;
    int d, E, Ep, T, mt, ksplit, nsplit;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem&) { return p.mt * p.nsplit; }
  __device__ static Job job(const Params& p, const SegSmem&, int t) {
    Job j;
    const int split = t / p.mt;
    j.m0 = (t - split * p.mt) * kBM;
    j.n0 = 0;
    j.seg = 0;
    j.sub = split;
    j.kbase = split * p.ksplit;
    const int rows = max(0, min(p.ksplit, p.T - j.kbase));
    j.kiters = (rows + kBK - 1) / kBK;
    j.idesc = idesc_bf16(128, p.Ep, true, true);
    return j;
  }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmX); tma_prefetch(&p.tmDL); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint64_t* bar) {
    const int row = j.kbase + kit * kBK;
    tma_load_2d(st, &p.tmX, bar, j.m0, row);
    tma_load_2d(st + kBox, &p.tmX, bar, j.m0 + 64, row);
#pragma unroll
    for (int i = 0; i < NB; ++i) tma_load_2d(st + (2 + i) * kBox, &p.tmDL, bar, 64 * i, row);
  }
  __device__ static void mma(const Job& j, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)
      umma_bf16(dt, sdesc_mnmajor(sa + kk * 2048, kBox), sdesc_mnmajor(sa + 2 * kBox + kk * 2048, kBox),
                j.idesc, (kit | kk) != 0);
  }
  // Row m of the partial, E floats from part + (split d + m) E: 16-byte stores when the rows are
  // 16-byte aligned (E a multiple of 4; a group of four is then wholly below E or wholly past it).
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int, int) {
    const int m = j.m0 + row;
    float* out = p.part + ((size_t)j.sub * p.d + (m < p.d ? m : 0)) * p.E;
    const bool vec = (p.E & 3) == 0;
#pragma unroll 1
    for (int c = 0; c < p.Ep; c += 32) {
      uint32_t v[32];
      tmem_ld32(ta + c, v);
      tmem_ld_wait();
      if (m >= p.d) continue;
      if (vec) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (c + 4 * q < p.E)
            *reinterpret_cast<float4*>(out + c + 4 * q) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                            __uint_as_float(v[4 * q + 3]));
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c + i < p.E) out[c + i] = __uint_as_float(v[i]);
      }
    }
  }
  // a split with no tokens contributes zeros
  __device__ static void epilogue_zero(const Params& p, const Job& j, int row, int) {
    const int m = j.m0 + row;
    if (m >= p.d) return;
    float* out = p.part + ((size_t)j.sub * p.d + m) * p.E;
    for (int e = 0; e < p.E; ++e) out[e] = 0.f;
  }
};

// The router's share of the input gradient on the tensor cores: r[t] = dl[t] W_r^T (M = 128
// tokens, N = 256 columns of d_model, K = E padded to 64, both operands bf16 K-major), stored as
// bf16 [T, d] for the token-owner combine that adds the expert rows.  With K this short the kernel
// is its output stores: two epilogue warps per TMEM lane quarter each store half of the columns.
struct RouterDx : PolicyDefaults {
  static constexpr int kId = kKRouterDx;
  static constexpr int kEpiWarps = 8;
  static constexpr int kStages = 3;
  static constexpr uint32_t kStageBytes = kTileA + 2 * kTileA;   // dl tile + W_r tile (256 rows)
  static constexpr int kAccCols = 256;
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdesc = idesc_bf16(128, 256, false, false);
  static constexpr uint32_t kEpiWarpBytes = 2 * 2048;   // two TMA-store boxes
  struct Params {
    CUtensorMap tmDL, tmWR, tmR;
    int T, d, mt, nt, kiters;
    Hdr* hdr;
    const Tables* tabs;
  };
  __device__ static int num_tiles(const Params& p, const SegSmem&) { return p.mt * p.nt; }
  __device__ static Job job(const Params& p, const SegSmem&, int t) {
    Job j;
    const int n = t / p.mt;
    j.m0 = (t - n * p.mt) * kBM;
    j.n0 = n * 256;
    j.seg = 0;
    j.sub = 0;
    j.kbase = 0;
    j.kiters = p.kiters;
    j.idesc = kIdesc;
    return j;
  }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmDL); tma_prefetch(&p.tmWR); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint64_t* bar) {
    tma_load_2d(st, &p.tmDL, bar, kit * kBK, j.m0);
    tma_load_2d(st + kTileA, &p.tmWR, bar, kit * kBK, j.n0);
  }
  __device__ static void mma(const Job&, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk)
      umma_bf16(dt, sdesc_kmajor(sa + kk * 32), sdesc_kmajor(sa + kTileA + kk * 32), kIdesc,
                (kit | kk) != 0);
  }
  __device__ static void epilogue(const Params& p, const Job& j, uint32_t ta, int row, int part, int,
                                  uint8_t* ebuf) {
    const int y = j.m0 + (row & ~31);
    if (y >= p.T) return;   // the tile's last warps may lie past the tokens
    store_acc_boxes(&p.tmR, y, j.n0, p.d, ta, row & 31, ebuf, 128 * part, 128 * part + 128);
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// Router logits on the tensor cores: l = x W_r with W_r split into three bf16 parts
// (W = hi + mid + lo, equal to W within fp32 rounding) stored K-major as [3][Ep][d_model].  x is
// exactly bf16, so every partial product is exact and only the accumulation rounds.  A tensor-core
// accumulator can lose about one fp32 unit of its own size per MMA step, so a single accumulator
// over all 3 d_model / 16 steps drifts by ~1e-5 of the logit at d_model = 2048.  K is therefore cut
// into chunks of kChunkKits 64-wide blocks; each chunk starts two fresh accumulators, one for the hi
// products (16 MMA steps) and one for the mid + lo products (2^8 smaller, so their rounding is
// negligible), and the epilogue adds both into fp32 registers.  A job is one (128-token tile, K
// chunk); the chunks of a tile run on one CTA, in order.  M = 128 tokens, N = Ep (64 or 128).
// After the last chunk the epilogue stores each lane's sums into the hi columns of the accumulator
// it still holds, then reads its logits back in 32-column pieces:
//   forward (kBwd = false): online softmax (running max and rescaled sum of exp) and the top-k
//     kept sorted while streaming, larger logit first and a tie keeping the lower expert index
//     (k <= 8); gates are p of the selected experts, or renormalised over them; logits written when
//     requested.
//   backward: a second pass gives dl_e = p_e (dg_slot(e) [e selected] - sum_j dg_j g_j) in fp32
//     and as the bf16 operand row (zero-padded to Ep), and for db one partial sum per warp of 32
//     tokens (summed in a fixed order afterwards).
constexpr int kRouterTopK = 8;

template <bool kBwd, bool kSplit>
struct RouterLogits : PolicyDefaults {
  static constexpr int kId = kBwd ? kKRouterDlogits : kKRoute;
  static constexpr int kEpiWarps = kSplit ? 8 : 4;       // kSplit: two per TMEM lane quarter
  static constexpr uint32_t kEpiWarpBytes = kSplit ? 3072 : 0;   // each warp's exchange buffer
  static constexpr int kStages = 3;
  static constexpr uint32_t kStageBytes = 4 * kTileA;   // x tile + three W_r parts (128 rows each)
  static constexpr int kAccCols = 256;                   // hi products, then mid + lo at +128
  static constexpr int kAccBufs = 2;
  static constexpr int kTmemCols = 512;
  static constexpr int kChunkKits = 4;                   // 256 of K per chunk
  static constexpr bool kStateful = true;
  struct Params {
    CUtensorMap tmX, tmW;
    const float* b_r;
    int T, d, E, Ep, k, renorm, mt, nch;
    int32_t* idx;            // forward output / backward input
    float* gates;            // forward output / backward input
    float* logits;           // forward, nullable
    const float* dgates;     // backward
    float* dlogits;          // backward
    uint16_t* dl_bf16;       // backward [T, Ep]
    float* db_part;          // backward [4 * mt, E]
    Hdr* hdr;
    const Tables* tabs;
  };
  // CTA b runs tiles b, b + grid, ... and each tile's nch chunks back to back
  __device__ static int num_tiles(const Params& p, const SegSmem&) {
    const int g = (int)gridDim.x;
    return g * ((p.mt + g - 1) / g) * p.nch;
  }
  __device__ static Job job(const Params& p, const SegSmem&, int t) {
    const int g = (int)gridDim.x;
    const int i = t / g;
    const int tile = (t - i * g) + (i / p.nch) * g;
    const int ch = i % p.nch;
    Job j;
    j.m0 = tile * kBM;
    j.n0 = 0;
    j.seg = 0;
    j.sub = ch;
    j.kbase = ch * kChunkKits;
    j.kiters = tile < p.mt ? min(kChunkKits, p.d / kBK - j.kbase) : 0;
    j.idesc = idesc_bf16(128, p.Ep, false, false);
    return j;
  }
  __device__ static void prefetch(const Params& p) { tma_prefetch(&p.tmX); tma_prefetch(&p.tmW); }
  __device__ static void load(const Params& p, const Job& j, int kit, uint8_t* st, uint64_t* bar) {
    const int kx = (j.kbase + kit) * kBK;
    tma_load_2d(st, &p.tmX, bar, kx, j.m0);
#pragma unroll
    for (int q = 0; q < 3; ++q) tma_load_3d(st + (1 + q) * kTileA, &p.tmW, bar, kx, 0, q);
  }
  // The hi and mid parts sit in adjacent 128-row slots (rows past Ep are TMA zero fill), so one
  // N = 256 MMA covers both and lands hi in columns [0, Ep) and mid in [128, 128 + Ep); lo then
  // accumulates onto mid.  Two MMAs per 16-deep step instead of three: the router is bound by MMA
  // issue, not by the tensor pipe.
  static constexpr uint32_t kIdescHiMid = idesc_bf16(128, 256, false, false);
  __device__ static void mma(const Job& j, int kit, uint32_t sa, uint32_t dt, int) {
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      const uint64_t da = sdesc_kmajor(sa + kk * 32);
      const bool acc = (kit | kk) != 0;
      umma_bf16(dt, da, sdesc_kmajor(sa + kTileA + kk * 32), kIdescHiMid, acc);
      umma_bf16(dt + 128, da, sdesc_kmajor(sa + 3 * kTileA + kk * 32), j.idesc, true);
    }
  }
  // kSplit (Ep = 128): eight epilogue warps, two per TMEM lane quarter; part h of a quarter sums and
  // finishes experts [64 h, 64 h + 64) of its 32 tokens, and the two parts meet in shared memory
  // (row maxima, sums of exp, top-k lists) before the outputs.  With one warp per quarter the last
  // slice's softmax and top-k over 128 experts took ~16 us a tile, one token per lane, while its
  // accumulator was held (split: 10-16% off the E = 128 routers; at Ep = 64 the second part would
  // have no experts, so those routers keep one warp per quarter).
  static constexpr int kPartCols = kSplit ? 64 : 128;
  struct EpiState {
    float l[kPartCols];   // this lane's running sums over the slices so far (its part)
    uint32_t xphase = 0;  // phase of the quarter's exchange barrier
  };
  static constexpr uint32_t kBarOff = 2560;   // the exchange barrier, in the part-0 warp's buffer
  static_assert(!kSplit || ((2 + 2 * kRouterTopK) * 32 * 4 <= kBarOff && kBarOff + 8 <= kEpiWarpBytes),
                "the exchange and its barrier fit the warp's buffer");
  // thread 0, before the kernel's first barrier fence: one two-arrival barrier per quarter
  __device__ static void init_epi(uint8_t* epi) {
    if constexpr (kSplit)
      for (int w = 0; w < 4; ++w) mbar_init(reinterpret_cast<uint64_t*>(epi + w * kEpiWarpBytes + kBarOff), 2);
  }
  __device__ static void epilogue_s(const Params& p, const Job& j, uint32_t ta, int row, int part, int,
                                    EpiState& st, uint8_t* ebuf) {
    const bool first = j.sub == 0;
    const int cb = part * kPartCols;
#pragma unroll
    for (int c = 0; c < kPartCols; c += 32) {
      if (cb + c < p.Ep) {   // warp-uniform: tcgen05.ld is warp-wide
        uint32_t h[32], r[32];
        tmem_ld32(ta + cb + c, h);
        tmem_ld32(ta + 128 + cb + c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          st.l[c + i] = (first ? 0.f : st.l[c + i]) + (__uint_as_float(h[i]) + __uint_as_float(r[i]));
      }
    }
    if (j.sub != p.nch - 1) return;
    // last slice: the sums go back into this accumulator's hi columns for the rolled passes below
#pragma unroll
    for (int c = 0; c < kPartCols; c += 32) {
      if (cb + c < p.Ep) {
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(st.l[c + i]);
        tmem_st32(ta + cb + c, v);
      }
    }
    tmem_st_wait();
    finish(p, j, ta, row, part, ebuf, st.xphase);
  }
  // logits of columns [c, c + 32) for this lane's token from S (bias added, -inf past E)
  __device__ static void chunk(const Params& p, uint32_t sum, int c, float (&l)[32]) {
    uint32_t v[32];
    tmem_ld32(sum + c, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = c + i;
      l[i] = e < p.E ? __uint_as_float(v[i]) + (p.b_r != nullptr ? p.b_r[e] : 0.f) : -INFINITY;
    }
  }
  // Logits [c, c + 32) of token t: 16-byte stores when the rows are 16-byte aligned (E a multiple
  // of 4, so a group of four is wholly below E or wholly past it), else one value at a time.
  __device__ static void store_logits(const Params& p, int t, int c, const float (&l)[32]) {
    float* row = p.logits + (size_t)t * p.E;
    if ((p.E & 3) == 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c + 4 * q < p.E)
          *reinterpret_cast<float4*>(row + c + 4 * q) =
              make_float4(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c + i < p.E) row[c + i] = l[i];
    }
  }
  // The two parts of a quarter (warps 4 apart) meet on a barrier of two arrivals, one per warp,
  // after each warp's shared-memory writes; the wait is bounded, so a partner that gave up leaves
  // an error instead of a hang.
  __device__ static void pair_sync(const Params& p, uint8_t* ebuf, int part, uint32_t& phase) {
    uint64_t* bar = reinterpret_cast<uint64_t*>((part == 0 ? ebuf : ebuf - 4 * kEpiWarpBytes) + kBarOff);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait_drain(bar, phase, wait_limit_ns(p.hdr));
    phase ^= 1u;
    if (!ok && (threadIdx.x & 31) == 0) record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmEpilogue);
  }
  __device__ static void finish(const Params& p, const Job& j, uint32_t sum, int row, int part, uint8_t* ebuf,
                                uint32_t& xphase) {
    const int t = j.m0 + row;
    const bool live = t < p.T;
    const int lane = threadIdx.x & 31;
    const int cb = part * kPartCols;
    // pass 1 over this part's experts: running max and rescaled sum of exp, and (forward) the top-k
    // kept sorted, larger logit first and a tie keeping the lower expert index
    float m = -INFINITY, z = 0.f;
    float tv[kRouterTopK];
    int ti[kRouterTopK];
#pragma unroll
    for (int s = 0; s < kRouterTopK; ++s) {
      tv[s] = -INFINITY;
      ti[s] = 0x7fffffff;
    }
#pragma unroll 1
    for (int c = cb; c < cb + kPartCols && c < p.Ep; c += 32) {
      float l[32];
      chunk(p, sum, c, l);
      float cm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) cm = fmaxf(cm, l[i]);
      if (cm > m) {
        z = (m == -INFINITY) ? 0.f : z * expf(m - cm);
        m = cm;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) z += (c + i < p.E) ? expf(l[i] - m) : 0.f;
      if (!kBwd) {
        if (live && p.logits != nullptr) store_logits(p, t, c, l);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float cv = l[i];
          int ci = c + i;
#pragma unroll
          for (int s = 0; s < kRouterTopK; ++s)
            if (cv > tv[s]) {
              const float fv = tv[s];
              const int fi = ti[s];
              tv[s] = cv;
              ti[s] = ci;
              cv = fv;
              ci = fi;
            }
        }
      }
    }
    if constexpr (kSplit) {
      // exchange with the other part of this quarter: word w of lane l at word w * 32 + l (the two
      // warps' buffers are 4 warps apart)
      float* mine = reinterpret_cast<float*>(ebuf);
      const float* other = reinterpret_cast<const float*>(part == 0 ? ebuf + 4 * kEpiWarpBytes : ebuf - 4 * kEpiWarpBytes);
      mine[0 * 32 + lane] = m;
      mine[1 * 32 + lane] = z;
      if (!kBwd) {
#pragma unroll
        for (int s = 0; s < kRouterTopK; ++s) {
          mine[(2 + s) * 32 + lane] = tv[s];
          mine[(2 + kRouterTopK + s) * 32 + lane] = __int_as_float(ti[s]);
        }
      }
      pair_sync(p, ebuf, part, xphase);
      const float mo = other[0 * 32 + lane], zo = other[1 * 32 + lane];
      float ov[kRouterTopK];
      int oi[kRouterTopK];
      if (!kBwd) {
#pragma unroll
        for (int s = 0; s < kRouterTopK; ++s) {
          ov[s] = other[(2 + s) * 32 + lane];
          oi[s] = __float_as_int(other[(2 + kRouterTopK + s) * 32 + lane]);
        }
      }
      pair_sync(p, ebuf, part, xphase);   // both have read before either buffer is written again
      // the token's max and sum of exp over all experts
      const float M = fmaxf(m, mo);
      z = (m == -INFINITY ? 0.f : z * expf(m - M)) + (mo == -INFINITY ? 0.f : zo * expf(mo - M));
      m = M;
      if (!kBwd) {
        // part 0's list (the lower expert indices) with part 1's entries inserted after equal ones
        if (part == 1) {
#pragma unroll
          for (int s = 0; s < kRouterTopK; ++s) {
            const float fv = tv[s];
            const int fi = ti[s];
            tv[s] = ov[s];
            ti[s] = oi[s];
            ov[s] = fv;
            oi[s] = fi;
          }
        }
#pragma unroll
        for (int q = 0; q < kRouterTopK; ++q) {
          float cv = ov[q];
          int ci = oi[q];
#pragma unroll
          for (int s = 0; s < kRouterTopK; ++s)
            if (cv > tv[s]) {
              const float fv = tv[s];
              const int fi = ti[s];
              tv[s] = cv;
              ti[s] = ci;
              cv = fv;
              ci = fi;
            }
        }
      }
    }
    if (!kBwd) {
      if (!live || part != 0) return;
      float zsel = 0.f;
#pragma unroll
      for (int s = 0; s < kRouterTopK; ++s)
        if (s < p.k) zsel += expf(tv[s] - m);
      const float denom = p.renorm ? zsel : z;
#pragma unroll
      for (int s = 0; s < kRouterTopK; ++s)
        if (s < p.k) {
          p.idx[(size_t)t * p.k + s] = ti[s];
          p.gates[(size_t)t * p.k + s] = expf(tv[s] - m) / denom;
        }
      return;
    }
    // backward pass 2: dl for every expert of this part
    float sdg = 0.f;
    int sid[kRouterTopK];
    float sgd[kRouterTopK];
#pragma unroll
    for (int s = 0; s < kRouterTopK; ++s) {
      sid[s] = -1;
      sgd[s] = 0.f;
      if (live && s < p.k) {
        sid[s] = p.idx[(size_t)t * p.k + s];
        sgd[s] = p.dgates[(size_t)t * p.k + s];
        sdg += sgd[s] * p.gates[(size_t)t * p.k + s];
      }
    }
    const int wq = row >> 5;   // TMEM lane quarter: one db partial per 32 tokens
#pragma unroll 1
    for (int c = cb; c < cb + kPartCols && c < p.Ep; c += 32) {
      float l[32];
      chunk(p, sum, c, l);
      float dl[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = c + i;
        float dsel = 0.f;
#pragma unroll
        for (int s = 0; s < kRouterTopK; ++s) dsel += (sid[s] == e) ? sgd[s] : 0.f;
        dl[i] = (live && e < p.E) ? expf(l[i] - m) / z * (dsel - sdg) : 0.f;
      }
      if (live) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(dl[2 * i], dl[2 * i + 1]);
        uint4* db = reinterpret_cast<uint4*>(p.dl_bf16 + (size_t)t * p.Ep + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) db[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c + i < p.E) p.dlogits[(size_t)t * p.E + c + i] = dl[i];
      }
      // db partial of these 32 tokens: a warp sum per expert, lane i keeps expert c + i
      float mine_db = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float v = dl[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == i) mine_db = v;
      }
      if (c + lane < p.E) p.db_part[((size_t)(j.m0 / kBM) * 4 + wq) * p.E + c + lane] = mine_db;
    }
  }
  __device__ static void epilogue_zero(const Params&, const Job&, int, int) {}
};

// ---------------------------------------------------------------------------------------------
// The persistent warp-specialised kernel
// ---------------------------------------------------------------------------------------------

template <class P>
constexpr size_t epi_bytes() {
  static_assert(P::kEpiWarpBytes % 1024 == 0, "boxes stay 1024-aligned");
  return (size_t)P::kEpiWarps * P::kEpiWarpBytes;
}

template <class P>
constexpr size_t smem_bytes() {
  static_assert(8 * (2 * P::kStages + 5) + 8 <= 256, "barriers fit their 256 bytes");
  return 1024 + (size_t)P::kStages * P::kStageBytes + epi_bytes<P>() + 256 + sizeof(SegSmem);
}

// Warps that copy gathered operand rows: warp 0 and, after the epilogue warps, three more.
constexpr int kGatherWarps = 4;

// producer, MMA, epilogue warps (+ the extra gather warps)
template <class P>
constexpr int threads_of() {
  return 64 + 32 * P::kEpiWarps + (P::kGather != 0 ? 32 * (kGatherWarps - 1) : 0);
}

template <class P>
__global__ void __launch_bounds__(threads_of<P>(), 1) gemm_kernel(const __grid_constant__ typename P::Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* epi = smem + (size_t)P::kStages * P::kStageBytes;   // per-warp epilogue shared memory
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + epi_bytes<P>());
  uint64_t* empty = full + P::kStages;
  uint64_t* tfull = empty + P::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;   // the MMA thread's last commit, waited for before TMEM is freed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  SegSmem& segs = *reinterpret_cast<SegSmem*>(epi + epi_bytes<P>() + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ClockSpan span;
  if (threadIdx.x == blockDim.x - 32) span.start();   // the last warp: off thread 0's setup path
  load_segs(segs, p.tabs);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], P::kEpiWarps);
    }
    mbar_init(drain, 1);
    if constexpr (P::kStateful) P::init_epi(epi);
    *abort_flag = 0;
    fence_mbar_init();
    P::prefetch(p);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, P::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = P::num_tiles(p, segs);
  const uint64_t limit = wait_limit_ns(p.hdr);

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int uses = 0;
      for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
        const Job j = P::job(p, segs, t);
        for (int kit = 0; kit < j.kiters; ++kit) {
          if (!mbar_wait(&empty[stage], phase ^ 1, limit, abort_flag)) {
            record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmProducer);
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], P::tx_bytes(j, kit, P::kStageBytes));
          P::load(p, j, kit, stages + (size_t)stage * P::kStageBytes, &full[stage]);
          ++uses;
          if (++stage == P::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every load this CTA issued lands before its shared memory is released (bounded)
      drain_fills(full, P::kStages, stage, phase, uses, limit);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int seq = 0;   // tiles with work issued by this CTA (the epilogue counts the same way)
      for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
        const Job j = P::job(p, segs, t);
        if (j.kiters == 0) continue;
        const int wait_at = P::acc_wait_kit(j);
        const uint32_t dt = tmem_base + (uint32_t)(acc * P::kAccCols);
        bool ok = true;
        for (int kit = 0; kit < j.kiters; ++kit) {
          if (kit == wait_at) {   // the epilogue must have released this accumulator
            if (!mbar_wait(&tempty[acc], acc_phase ^ 1, limit, abort_flag)) {
              record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmMma);
              *abort_flag = 1;
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!mbar_wait(&full[stage], phase, limit, abort_flag)) {
            record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          P::mma(j, kit, smem_u32(stages + (size_t)stage * P::kStageBytes), dt, seq);
          umma_commit(&empty[stage]);
          if (++stage == P::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        ++seq;
        if (++acc == P::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA this thread issued has completed before TMEM is freed (bounded)
      umma_commit(drain);
      mbar_wait_drain(drain, 0, limit);
    }
  } else {
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // column share when two warps serve one quarter
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    int seq = 0;
    typename P::EpiState es;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Job j = P::job(p, segs, t);
      if (j.kiters == 0) {
        if (part == 0) P::epilogue_zero(p, j, row, part);
        continue;
      }
      if (!mbar_wait_idle(&tfull[acc], acc_phase, limit, abort_flag)) {
        record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t ta = tmem_base + (uint32_t)(acc * P::kAccCols) + ((uint32_t)(q * 32) << 16);
      if constexpr (P::kStateful)
        P::epilogue_s(p, j, ta, row, part, seq, es, epi + (size_t)(warp - 2) * P::kEpiWarpBytes);
      else if constexpr (P::kEpiWarpBytes > 0)
        P::epilogue(p, j, ta, row, part, seq, epi + (size_t)(warp - 2) * P::kEpiWarpBytes);
      else
        P::epilogue(p, j, ta, row, part, seq);
      ++seq;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == P::kAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();   // this warp's output stores (if any) have landed
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == blockDim.x - 32) span.stop(P::kId);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, P::kTmemCols);
  }
}

// The CTA-pair version: a cluster of two CTAs shares every tile.  Both CTAs run the producer and
// the epilogue for their own 128 rows; only the even CTA's MMA thread issues (cta_group::2):
//   full[s]    even CTA: one expect_tx arrival, completed by both CTAs' TMA bytes
//   empty[s]   even CTA: freed by a commit of the MMA thread once the slot's MMAs are done; odd
//              CTA: freed by the even CTA's producer, which forwards that completion (a relaxed
//              remote arrival, after its own loads) when it refills the slot.  One commit per
//              slot: a second commit per 64-wide K block cost 6-8% of the MMA rate (measured in
//              SM cycles), while slots of two K blocks, with half the slots, lost more to the
//              shallower pipeline.
//   tfull[a]   each CTA: the finished accumulator, committed by the MMA thread to both CTAs
//   tempty[a]  even CTA: released by the epilogue warps of both CTAs (remote arrivals)
// Both CTAs walk the same tile sequence (pair id, stride = number of pairs).  Every wait is
// bounded; whatever happens, both CTAs meet at the final cluster barrier before TMEM is freed, so
// neither exits while the other may still touch its shared memory.
template <class P>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_of<P>(), 1)
    gemm_pair_kernel(const __grid_constant__ typename P::Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* epi = smem + (size_t)P::kStages * P::kStageBytes;   // 1024-aligned staging boxes
  uint64_t* full = reinterpret_cast<uint64_t*>(epi + epi_bytes<P>());
  uint64_t* empty = full + P::kStages;
  uint64_t* tfull = empty + P::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;   // the MMA thread's last commit, waited for before TMEM is freed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  SegSmem& segs = *reinterpret_cast<SegSmem*>(epi + epi_bytes<P>() + 256);

  constexpr int kSub = P::kSub;
  constexpr int kSlots = P::kStages / kSub;
  constexpr size_t kSlotBytes = (size_t)kSub * P::kStageBytes;
  static_assert(P::kStages % kSub == 0, "whole slots");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  ClockSpan span;
  if (threadIdx.x == blockDim.x - 32) span.start();   // the last warp: off thread 0's setup path
  load_segs(segs, p.tabs);
  if (threadIdx.x == 0) {
    for (int s = 0; s < P::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * P::kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    P::prefetch(p);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, P::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = P::num_tiles(p, segs);
  const uint64_t limit = wait_limit_ns(p.hdr);

  if (warp == 0 && P::kGather == 0) {
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      int uses = 0;   // slots filled so far; from kSlots on, every fill follows a completed use
      // test hook: the first pair skips one fill (no loads, no expected bytes), so that the MMA
      // thread's wait for it runs out
      const int skip = pair == 0 ? *((volatile const int32_t*)&p.hdr->stall_fill_p1) - 1 : -1;
      for (int t = pair; t < ntiles && !*abort_flag; t += npairs) {
        const Job j = P::job(p, segs, t);
        for (int k0 = 0; k0 < j.kiters; k0 += kSub) {
          if (!mbar_wait(&empty[slot], phase ^ 1, limit, abort_flag)) {
            record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmProducer);
            *abort_flag = 1;
            break;
          }
          const int nsb = min(kSub, j.kiters - k0);
          if (uses != skip) {
            if (rank == 0) {
              uint32_t tx = 0;
              for (int sb = 0; sb < nsb; ++sb) tx += P::tx_bytes(j, k0 + sb, P::kStageBytes);
              mbar_arrive_expect_tx(&full[slot], 2 * tx);
            }
            uint8_t* st = stages + (size_t)slot * kSlotBytes;
            for (int sb = 0; sb < nsb; ++sb)
              P::load(p, j, k0 + sb, st + (size_t)sb * P::kStageBytes, cluster_addr(&full[slot], 0), rank);
          }
          if (rank == 0 && uses >= kSlots) mbar_arrive_cluster_relaxed(cluster_addr(&empty[slot], 1));
          ++uses;
          if (++slot == kSlots) {
            slot = 0;
            phase ^= 1;
          }
        }
      }
      // every load of the pair lands before either CTA's shared memory is released: the even CTA's
      // full barriers count both CTAs' bytes, and the odd CTA waits at the final cluster barrier
      // (bounded; a skipped fill never completes and ends this wait at its limit)
      if (rank == 0) drain_fills(full, kSlots, slot, phase, uses, limit);
    }
  } else if (warp == 0 || warp >= 2 + P::kEpiWarps) {
    if constexpr (P::kGather != 0) {
      // Gathered operand rows: four warps copy them, each 32 of the stage's 128 lines of 128 bytes,
      // with eight tile::gather4 copies of four lines (lanes 0..7).  A single warp issuing all 32
      // copies of a stage left the tensor pipe idle most of the time, and so did 16-byte cp.async
      // copies from one or four warps; four warps of gather4 copies halve that loss.  Warp 0 also
      // announces the pair's bytes, loads the other operand by TMA and forwards the slot's release
      // to the odd CTA.  Each lane holds the token of one line, fetched one tile (kGather 1) or
      // kAhead stages (kGather 2) ahead, and hands it round by shuffle.
      static_assert(kSub == 1, "gathered loads fill one K block per slot");
      constexpr int kAhead = 8;
      const bool lead = warp == 0;
      const int gw = lead ? 0 : warp - (1 + P::kEpiWarps);   // lines 32 gw .. 32 gw + 31
      int slot = 0;
      uint32_t phase = 0;
      int uses = 0;
      const int skip = pair == 0 ? *((volatile const int32_t*)&p.hdr->stall_fill_p1) - 1 : -1;
      bool ok = true;
      auto fill = [&](const Job& j, int kit, int tokv) {
        int w = 1;
        if (lane == 0) w = (*abort_flag == 0 && mbar_wait(&empty[slot], phase ^ 1, limit, abort_flag)) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, w, 0) == 0) {
          if (lane == 0) {
            record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmProducer);
            *abort_flag = 1;
          }
          ok = false;
          return;
        }
        if (uses != skip) {
          uint8_t* st = stages + (size_t)slot * kSlotBytes;
          if (lead && lane == 0) {
            if (rank == 0) mbar_arrive_expect_tx(&full[slot], 2 * P::tx_bytes(j, kit, P::kStageBytes));
            P::load(p, j, kit, st, cluster_addr(&full[slot], 0), rank);
          }
          // lane l < 8: lines 32 gw + 4 l .. + 3, whose tokens lanes 4 l .. 4 l + 3 hold
          const GatherOp op = P::gather_op(p, j, kit, rank);
          int4 r;
          r.x = __shfl_sync(0xffffffffu, tokv, (4 * lane + 0) & 31);
          r.y = __shfl_sync(0xffffffffu, tokv, (4 * lane + 1) & 31);
          r.z = __shfl_sync(0xffffffffu, tokv, (4 * lane + 2) & 31);
          r.w = __shfl_sync(0xffffffffu, tokv, (4 * lane + 3) & 31);
          if (lane < 8)
            tma_gather4_pair(smem_u32(st) + op.dst + (uint32_t)(32 * gw + 4 * lane) * 128u, op.map,
                             cluster_addr(&full[slot], 0), gw < 2 ? op.col0 : op.col1, r);
        }
        if (lead && lane == 0 && rank == 0 && uses >= kSlots) mbar_arrive_cluster_relaxed(cluster_addr(&empty[slot], 1));
        ++uses;
        if (++slot == kSlots) {
          slot = 0;
          phase ^= 1;
        }
      };
      if constexpr (P::kGather == 1) {
        // a tile's rows are the same for all its K blocks: fetch the next tile's with this one
        auto tile_tok = [&](int t) { return __ldg(P::gather_tok(p, P::job(p, segs, t), 0, rank) + 32 * gw + lane); };
        int next = 0;
        if (pair < ntiles) next = tile_tok(pair);
        for (int t = pair; t < ntiles && ok; t += npairs) {
          const Job j = P::job(p, segs, t);
          const int tokv = next;
          if (t + npairs < ntiles) next = tile_tok(t + npairs);
          for (int kit = 0; kit < j.kiters && ok; ++kit) fill(j, kit, tokv);
        }
      } else {
        // the K rows change every stage: a cursor over this pair's stages, in the order they are
        // filled, keeps kAhead stages' tokens in flight (the two 64-column boxes share the rows)
        int pt = pair, pkit = 0;
        Job pj{};
        if (pt < ntiles) pj = P::job(p, segs, pt);
        auto ahead = [&]() {
          while (pt < ntiles && pkit >= pj.kiters) {
            pt += npairs;
            pkit = 0;
            if (pt < ntiles) pj = P::job(p, segs, pt);
          }
          if (pt >= ntiles) return 0;
          const int v = __ldg(P::gather_tok(p, pj, pkit, rank) + 32 * (gw & 1) + lane);
          ++pkit;
          return v;
        };
        int ring[kAhead];
#pragma unroll
        for (int i = 0; i < kAhead; ++i) ring[i] = ahead();
        for (int t = pair; t < ntiles && ok; t += npairs) {
          const Job j = P::job(p, segs, t);
          for (int kit = 0; kit < j.kiters && ok; ++kit) {
            const int tokv = ring[0];
#pragma unroll
            for (int i = 0; i + 1 < kAhead; ++i) ring[i] = ring[i + 1];
            ring[kAhead - 1] = ahead();
            fill(j, kit, tokv);
          }
        }
      }
      // every load of the pair lands before either CTA's shared memory is released (as above)
      if (lead && lane == 0 && rank == 0) drain_fills(full, kSlots, slot, phase, uses, limit);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int slot = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int seq = 0;
      const Job j{};   // the pair problems' MMAs depend only on the K block
      for (int t = pair; t < ntiles && !*abort_flag; t += npairs) {
        // the tile's K blocks only: the single issuing thread bounds these kernels, and a full
        // job (segment search, divisions) between tiles leaves the tensor pipe idle
        const int kiters = P::mma_kiters(p, segs, t);
        if (kiters == 0) continue;
        const uint32_t dt = tmem_base + (uint32_t)(acc * P::kAccCols);
        // both CTAs' epilogues must have released this accumulator
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, limit, abort_flag)) {
          record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmMma);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int k0 = 0; k0 < kiters; k0 += kSub) {
          if (!mbar_wait(&full[slot], phase, limit, abort_flag)) {
            record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmMma);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsb = min(kSub, kiters - k0);
          const uint32_t sa = smem_u32(stages + (size_t)slot * kSlotBytes);
          for (int sb = 0; sb < nsb; ++sb) P::mma(j, k0 + sb, sa + sb * P::kStageBytes, dt, seq);
          umma_commit_pair(smem_u32(&empty[slot]));
          if (++slot == kSlots) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair(cluster_addr(&tfull[acc], 0));
        umma_commit_pair(cluster_addr(&tfull[acc], 1));
        ++seq;
        if (++acc == P::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every pair MMA issued has completed before either CTA frees its TMEM (bounded)
      umma_commit_pair(cluster_addr(drain, 0));
      mbar_wait_drain(drain, 0, limit);
    }
  } else {
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int part = (warp - 2) >> 2;  // column share when two warps serve one quarter
    const int row = q * 32 + lane;
    uint8_t* ebuf = epi + (size_t)(warp - 2) * P::kEpiWarpBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    int seq = 0;
    // epilogue-only tiles of this pair (pair, pair + npairs, ...), stored while an MMA tile is pending
    int zt = pair;
    int nzt = 0;
    if constexpr (P::kZeroTiles) nzt = P::zero_tiles(p, segs);
    auto zero_tile = [&]() {
      Job j = P::job(p, segs, ntiles + zt);
      j.m0 += kBM * rank;
      if (part == 0) P::epilogue_zero(p, j, row, part);
      zt += npairs;
    };
    for (int t = pair; t < ntiles; t += npairs) {
      Job j = P::job(p, segs, t);
      j.m0 += kBM * rank;   // this CTA's 128 rows of the pair tile
      if (j.kiters == 0) {
        if (part == 0) P::epilogue_zero(p, j, row, part);
        continue;
      }
      if constexpr (P::kZeroTiles) {   // one decision per warp: its tcgen05 loads below are warp-wide
        while (zt < nzt) {
          const int ready = lane == 0 ? (int)mbar_try_wait(&tfull[acc], acc_phase) : 0;
          if (__shfl_sync(0xffffffffu, ready, 0)) break;
          zero_tile();
        }
      }
      if (!mbar_wait_idle(&tfull[acc], acc_phase, limit, abort_flag)) {
        record_error(p.hdr, MOE_ERR_TIMEOUT, kSiteGemmEpilogue);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      P::epilogue(p, j, tmem_base + (uint32_t)(acc * P::kAccCols) + ((uint32_t)(q * 32) << 16), row, part,
                  seq, ebuf);
      ++seq;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[acc], 0));
      if (++acc == P::kAccBufs) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if constexpr (P::kZeroTiles) {
      while (zt < nzt && !*abort_flag) zero_tile();
    }
    if (lane == 0) bulk_wait_all();   // this warp's output stores have landed
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == blockDim.x - 32) span.stop(P::kId);
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, P::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side: tensor maps and launches
// ---------------------------------------------------------------------------------------------

template <class P>
cudaError_t launch(const typename P::Params& p, cudaStream_t s) {
  constexpr size_t smem = smem_bytes<P>();
  static_assert(smem <= 232448, "shared memory per block");
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_mark(P::kId, s, true);
  gemm_kernel<P><<<num_sms(), threads_of<P>(), smem, s>>>(p);
  prof_mark(P::kId, s, false);
  return cudaGetLastError();
}

// Pairs: as many clusters as fit at once (two CTAs each), one persistent pair per cluster slot.
template <class P>
cudaError_t launch_pair(const typename P::Params& p, cudaStream_t s) {
  constexpr size_t smem = smem_bytes<P>();
  static_assert(smem <= 232448, "shared memory per block");
  static int grid = 0;   // per problem type and process (all devices here are alike)
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (grid == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(threads_of<P>(), 1, 1);
    cfg.dynamicSmemBytes = smem;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, gemm_pair_kernel<P>, &cfg) != cudaSuccess || nclusters <= 0) {
      (void)cudaGetLastError();
      nclusters = num_sms() / 2;
    }
    grid = 2 * std::min(nclusters, num_sms() / 2);
  }
  prof_mark(P::kId, s, true);
  gemm_pair_kernel<P><<<grid, threads_of<P>(), smem, s>>>(p);
  prof_mark(P::kId, s, false);
  return cudaGetLastError();
}

}  // namespace

namespace {

template <bool kKeep, bool kG>
cudaError_t launch_gate_up(const Cfg& c, const Layout& L, const FfnFwdArgs& a, int keep, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  typename FwdGateUpT<kKeep, kG>::Params p1{};
  const bool mx = kG ? map_gather_rows(&p1.tmX, a.x_tok, c.d, c.T) : map_2d(&p1.tmX, a.x_perm, c.d, rows, 64, 128);
  p1.tok = a.tok;
  if (!mx ||
      !map_3d(&p1.tmWg, a.Wg, c.d, c.f, c.G, 64, 128) || !map_3d(&p1.tmWu, a.Wu, c.d, c.f, c.G, 64, 128) ||
      !map_2d(&p1.tmH, a.h, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  // the kept planes hold `keep` rows (in `saved`, or the workspace for granular calls)
  if (kKeep && (!map_2d(&p1.tmA, a.a_keep, c.f, (uint64_t)keep, 32, 32) ||
                !map_2d(&p1.tmB, a.b_keep, c.f, (uint64_t)keep, 32, 32)))
    return cudaErrorInvalidValue;
  p1.f = c.f;
  p1.d = c.d;
  p1.nt = (c.f + 127) / 128;
  p1.keep_rows = keep;
  p1.hdr = a.hdr;
  p1.tabs = a.tabs;
  return launch_pair<FwdGateUpT<kKeep, kG>>(p1, s);
}

// Weight gradients (bf16 operands in both the bf16 and the FP8 backward): dWg = dA^T X, dWu = dB^T X,
// dWd = dY^T Hg per expert.
// x and dY rows from x_perm / dy_perm, or (tok non-null) gathered from x / dy in token order.
template <bool kG>
cudaError_t launch_wgrad_t(const Cfg& c, const Layout& L, const uint16_t* dA, const uint16_t* dB, const uint16_t* Hg,
                           const uint16_t* x_rows, const uint16_t* dy_rows, const int32_t* tok, uint16_t* dWg,
                           uint16_t* dWu, uint16_t* dWd, Hdr* hdr, const Tables* tabs, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  typename WgradT<kG>::Params p4{};
  const bool tok_side = kG ? map_gather_rows(&p4.tmX, x_rows, c.d, c.T) && map_gather_rows(&p4.tmDY, dy_rows, c.d, c.T)
                           : map_mn2(&p4.tmX, x_rows, c.d, rows) && map_mn2(&p4.tmDY, dy_rows, c.d, rows);
  if (!tok_side || !map_mn2(&p4.tmDA, dA, c.f, rows) || !map_mn2(&p4.tmDB, dB, c.f, rows) ||
      !map_mn2(&p4.tmHg, Hg, c.f, rows) || !map_3d(&p4.tmdWg, dWg, c.d, c.f, c.G, 32, 32) ||
      !map_3d(&p4.tmdWu, dWu, c.d, c.f, c.G, 32, 32) || !map_3d(&p4.tmdWd, dWd, c.f, c.d, c.G, 32, 32))
    return cudaErrorInvalidValue;
  p4.tok = tok;
  p4.dWg = dWg;
  p4.dWu = dWu;
  p4.dWd = dWd;
  p4.f = c.f;
  p4.d = c.d;
  p4.mt_f = (c.f + kPairM - 1) / kPairM;
  p4.nt_d = (c.d + 255) / 256;
  p4.mt_d = (c.d + kPairM - 1) / kPairM;
  p4.nt_f = (c.f + 255) / 256;
  p4.tps = 2 * p4.mt_f * p4.nt_d + p4.mt_d * p4.nt_f;
  p4.hdr = hdr;
  p4.tabs = tabs;
  return launch_pair<WgradT<kG>>(p4, s);
}

cudaError_t launch_wgrad(const Cfg& c, const Layout& L, const uint16_t* dA, const uint16_t* dB, const uint16_t* Hg,
                         const uint16_t* x_rows, const uint16_t* dy_rows, const int32_t* tok, uint16_t* dWg,
                         uint16_t* dWu, uint16_t* dWd, Hdr* hdr, const Tables* tabs, cudaStream_t s) {
  return tok != nullptr ? launch_wgrad_t<true>(c, L, dA, dB, Hg, x_rows, dy_rows, tok, dWg, dWu, dWd, hdr, tabs, s)
                        : launch_wgrad_t<false>(c, L, dA, dB, Hg, x_rows, dy_rows, tok, dWg, dWu, dWd, hdr, tabs, s);
}

}  // namespace

cudaError_t launch_ffn_fwd(const Cfg& c, const Layout& L, const FfnFwdArgs& a, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  const int keep = (int)std::min<int64_t>(c.keep, L.rows);
  const bool g = a.tok != nullptr;   // x rows gathered from token order
  cudaError_t e = keep > 0 ? (g ? launch_gate_up<true, true>(c, L, a, keep, s) : launch_gate_up<true, false>(c, L, a, keep, s))
                           : (g ? launch_gate_up<false, true>(c, L, a, 0, s) : launch_gate_up<false, false>(c, L, a, 0, s));
  if (e != cudaSuccess) return e;
  FwdDown::Params p2{};
  if (!map_2d(&p2.tmH, a.h, c.f, rows, 64, 128) || !map_3d(&p2.tmWd, a.Wd, c.f, c.d, c.G, 64, 128) ||
      !map_2d(&p2.tmO, a.o_perm, c.d, rows, 32, 32))
    return cudaErrorInvalidValue;
  p2.f = c.f;
  p2.d = c.d;
  p2.nt = (c.d + 255) / 256;
  p2.hdr = a.hdr;
  p2.tabs = a.tabs;
  return launch_pair<FwdDown>(p2, s);
}

namespace {

// dY and x rows from dy_perm / x_perm, or (kG) gathered from dy / x in token order through a.tok.
template <bool kG>
cudaError_t launch_ffn_bwd_t(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  typename BwdDhT<kG>::Params p2{};
  const bool mdy = kG ? map_gather_rows(&p2.tmDY, a.dy_tok, c.d, c.T) : map_2d(&p2.tmDY, a.dy_perm, c.d, rows, 64, 128);
  if (!mdy || !map_mn2_g(&p2.tmWdT, a.Wd, c.f, c.d, c.G) || !map_2d(&p2.tmDH, a.dh, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  p2.tok = a.tok;
  p2.f = c.f;
  p2.d = c.d;
  p2.nt = (c.f + 255) / 256;
  p2.hdr = a.hdr;
  p2.tabs = a.tabs;
  cudaError_t e = launch_pair<BwdDhT<kG>>(p2, s);
  if (e != cudaSuccess) return e;
  const int keep = (int)std::min<int64_t>(c.keep, L.rows);
  if (keep > 0) {   // rows whose a, b the forward kept: an element-wise SwiGLU backward
    e = launch_swiglu_bwd_kept(c, L, a, s);
    if (e != cudaSuccess) return e;
  }

  typename BwdFusedT<kG>::Params p3{};
  const bool mx = kG ? map_gather_rows(&p3.tmX, a.x_tok, c.d, c.T) : map_2d(&p3.tmX, a.x_perm, c.d, rows, 64, 128);
  if (!mx || !map_3d(&p3.tmWg, a.Wg, c.d, c.f, c.G, 64, 128) ||
      !map_3d(&p3.tmWu, a.Wu, c.d, c.f, c.G, 64, 128) || !map_2d(&p3.tmDA, a.dA, c.f, rows, 32, 32) ||
      !map_2d(&p3.tmDB, a.dB, c.f, rows, 32, 32) || !map_2d(&p3.tmHg, a.Hg, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  p3.tok = a.tok;
  p3.DH = a.dh;
  p3.gate_of_prow = a.gate_of_prow;
  p3.dg_part = a.dg_part;
  p3.f = c.f;
  p3.d = c.d;
  p3.nt = L.ntf;
  p3.ndg = L.ndg;
  p3.keep_rows = keep;
  p3.hdr = a.hdr;
  p3.tabs = a.tabs;
  e = launch_pair<BwdFusedT<kG>>(p3, s);
  if (e != cudaSuccess) return e;

  e = launch_wgrad(c, L, a.dA, a.dB, a.Hg, kG ? a.x_tok : a.x_perm, kG ? a.dy_tok : a.dy_perm, kG ? a.tok : nullptr,
                   a.dWg, a.dWu, a.dWd, a.hdr, a.tabs, s);
  if (e != cudaSuccess) return e;

  DgradX::Params p5{};
  if (!map_2d(&p5.tmDA, a.dA, c.f, rows, 64, 128) || !map_2d(&p5.tmDB, a.dB, c.f, rows, 64, 128) ||
      !map_mn2_g(&p5.tmWgT, a.Wg, c.d, c.f, c.G) || !map_mn2_g(&p5.tmWuT, a.Wu, c.d, c.f, c.G) ||
      !map_2d(&p5.tmDX, a.dx_perm, c.d, rows, 32, 32))
    return cudaErrorInvalidValue;
  p5.f = c.f;
  p5.d = c.d;
  p5.nt = (c.d + 255) / 256;
  p5.hdr = a.hdr;
  p5.tabs = a.tabs;
  return launch_pair<DgradX>(p5, s);
}

}  // namespace

cudaError_t launch_ffn_bwd(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s) {
  return a.tok != nullptr ? launch_ffn_bwd_t<true>(c, L, a, s) : launch_ffn_bwd_t<false>(c, L, a, s);
}

cudaError_t launch_gate_up_fp8(const Cfg& c, const Layout& L, const GateUpFp8Args& a, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  FwdGateUp8::Params p{};
  if (!map_u8_2d(&p.tmX, a.x8, c.d, rows) || !map_u8_3d(&p.tmWg, a.wg8, c.d, c.f, c.G) ||
      !map_u8_3d(&p.tmWu, a.wu8, c.d, c.f, c.G) || !map_2d(&p.tmH, a.h, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  p.xs = a.xs;
  p.gs = a.gs;
  p.us = a.us;
  p.f = c.f;
  p.d = c.d;
  p.nt = (c.f + 127) / 128;
  p.hdr = a.hdr;
  p.tabs = a.tabs;
  return launch_pair<FwdGateUp8>(p, s);
}

cudaError_t launch_down_fp8(const Cfg& c, const Layout& L, const DownFp8Args& a, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  FwdDown8::Params p{};
  if (!map_u8_2d(&p.tmA, a.h8, c.f, rows) || !map_u8_3d(&p.tmB, a.wd8, c.f, c.d, c.G) ||
      !map_2d(&p.tmO, a.o, c.d, rows, 32, 32))
    return cudaErrorInvalidValue;
  p.as = a.hs;
  p.bs = a.ds;
  p.K = c.f;
  p.N = c.d;
  p.nt = (c.d + 255) / 256;
  p.hdr = a.hdr;
  p.tabs = a.tabs;
  return launch_pair<FwdDown8>(p, s);
}

// The FP8 backward of the expert FFN (reading in moe.h): dh' = dY8 WdT8^T (e4m3, bf16 out); the
// recompute of a, b from the forward's codes with the SwiGLU backward (dA, dB, Hg bf16); the bf16
// weight gradients; the joined [dA | dB] rows quantised per row; dX = dAB8 WguT8^T (e4m3).
cudaError_t launch_ffn_bwd_fp8(const Cfg& c, const Layout& L, const FfnBwd8Args& a, cudaStream_t s) {
  const uint64_t rows = (uint64_t)L.rows;
  BwdDh8::Params p1{};
  if (!map_u8_2d(&p1.tmA, a.dy8, c.d, rows) || !map_u8_3d(&p1.tmB, a.wdt8, c.d, c.f, c.G) ||
      !map_2d(&p1.tmO, a.dh, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  p1.as = a.dys;
  p1.bs = a.wdts;
  p1.K = c.d;
  p1.N = c.f;
  p1.nt = (c.f + 255) / 256;
  p1.hdr = a.hdr;
  p1.tabs = a.tabs;
  cudaError_t e = launch_pair<BwdDh8>(p1, s);
  if (e != cudaSuccess) return e;

  BwdFused8::Params p2{};
  if (!map_u8_2d(&p2.tmX, a.x8, c.d, rows) || !map_u8_3d(&p2.tmWg, a.wg8, c.d, c.f, c.G) ||
      !map_u8_3d(&p2.tmWu, a.wu8, c.d, c.f, c.G) || !map_2d(&p2.tmDA, a.dA, c.f, rows, 32, 32) ||
      !map_2d(&p2.tmDB, a.dB, c.f, rows, 32, 32) || !map_2d(&p2.tmHg, a.Hg, c.f, rows, 32, 32))
    return cudaErrorInvalidValue;
  p2.xs = a.xs;
  p2.gs = a.gs;
  p2.us = a.us;
  p2.DH = a.dh;
  p2.gate_of_prow = a.gate_of_prow;
  p2.dg_part = a.dg_part;
  p2.f = c.f;
  p2.d = c.d;
  p2.nt = L.ntf;
  p2.ndg = L.ndg;
  p2.hdr = a.hdr;
  p2.tabs = a.tabs;
  e = launch_pair<BwdFused8>(p2, s);
  if (e != cudaSuccess) return e;

  e = launch_wgrad(c, L, a.dA, a.dB, a.Hg, a.x_perm, a.dy_perm, nullptr, a.dWg, a.dWu, a.dWd, a.hdr, a.tabs, s);
  if (e != cudaSuccess) return e;
  e = launch_quantize_rows2_e4m3(a.dA, c.f, a.dB, c.f, (int64_t)rows, a.dab8, a.dabs, s, a.tabs);
  if (e != cudaSuccess) return e;

  DgradX8::Params p3{};
  if (!map_u8_2d(&p3.tmA, a.dab8, 2 * c.f, rows) || !map_u8_3d(&p3.tmB, a.wgut8, 2 * c.f, c.d, c.G) ||
      !map_2d(&p3.tmO, a.dx_perm, c.d, rows, 32, 32))
    return cudaErrorInvalidValue;
  p3.as = a.dabs;
  p3.bs = a.wguts;
  p3.K = 2 * c.f;
  p3.N = c.d;
  p3.nt = (c.d + 255) / 256;
  p3.hdr = a.hdr;
  p3.tabs = a.tabs;
  return launch_pair<DgradX8>(p3, s);
}

template <int NB>
cudaError_t launch_router_dwr_nb(const Cfg& c, const Layout& L, const uint16_t* x, const uint16_t* dl_bf16,
                                 float* dwr_part, Hdr* hdr, const Tables* tabs, cudaStream_t s) {
  typename RouterDwrT<NB>::Params p{};
  if (!map_2d(&p.tmX, x, c.d, c.T, 64, 64) || !map_2d(&p.tmDL, dl_bf16, L.Ep, c.T, 64, 64))
    return cudaErrorInvalidValue;
  p.part = dwr_part;
  p.d = c.d;
  p.E = c.E;
  p.Ep = L.Ep;
  p.T = c.T;
  p.mt = (c.d + kBM - 1) / kBM;
  p.nsplit = L.nsplit_dwr;
  p.ksplit = router_dwr_ksplit(c.T, L.nsplit_dwr);
  p.hdr = hdr;
  p.tabs = tabs;
  return launch<RouterDwrT<NB>>(p, s);
}

cudaError_t launch_router_dwr(const Cfg& c, const Layout& L, const uint16_t* x, const uint16_t* dl_bf16,
                              float* dwr_part, Hdr* hdr, const Tables* tabs, cudaStream_t s) {
  switch (L.Ep / 64) {
    case 1: return launch_router_dwr_nb<1>(c, L, x, dl_bf16, dwr_part, hdr, tabs, s);
    case 2: return launch_router_dwr_nb<2>(c, L, x, dl_bf16, dwr_part, hdr, tabs, s);
    case 3: return launch_router_dwr_nb<3>(c, L, x, dl_bf16, dwr_part, hdr, tabs, s);
    default: return launch_router_dwr_nb<4>(c, L, x, dl_bf16, dwr_part, hdr, tabs, s);
  }
}

template <bool kBwd, bool kSplit>
cudaError_t launch_router_tc_t(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s) {
  using P = RouterLogits<kBwd, kSplit>;
  typename P::Params p{};
  if (!map_2d(&p.tmX, a.x, c.d, c.T, 64, 128) || !map_3d(&p.tmW, a.wr3, c.d, L.Ep, 3, 64, 128))
    return cudaErrorInvalidValue;
  p.b_r = a.b_r;
  p.T = c.T;
  p.d = c.d;
  p.E = c.E;
  p.Ep = L.Ep;
  p.k = c.k;
  p.renorm = c.renorm;
  p.mt = (c.T + kBM - 1) / kBM;
  p.nch = (c.d / kBK + P::kChunkKits - 1) / P::kChunkKits;
  p.idx = a.idx;
  p.gates = a.gates;
  p.logits = a.logits;
  p.dgates = a.dgates;
  p.dlogits = a.dlogits;
  p.dl_bf16 = a.dl_bf16;
  p.db_part = a.db_part;
  p.hdr = a.hdr;
  p.tabs = a.tabs;
  return launch<P>(p, s);
}

template <bool kBwd>
cudaError_t launch_router_tc(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s) {
  return L.Ep > 64 ? launch_router_tc_t<kBwd, true>(c, L, a, s) : launch_router_tc_t<kBwd, false>(c, L, a, s);
}

cudaError_t launch_route_tc(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s) {
  return launch_router_tc<false>(c, L, a, s);
}

cudaError_t launch_router_dlogits_tc(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s) {
  return launch_router_tc<true>(c, L, a, s);
}

cudaError_t launch_router_dx(const Cfg& c, const Layout& L, const RouterDxArgs& a, cudaStream_t s) {
  RouterDx::Params p{};
  if (!map_2d(&p.tmDL, a.dl_bf16, L.Ep, c.T, 64, 128) || !map_2d(&p.tmWR, a.wr_bf16, L.Ep, c.d, 64, 256) ||
      !map_2d(&p.tmR, a.r, c.d, c.T, 32, 32))
    return cudaErrorInvalidValue;
  p.T = c.T;
  p.d = c.d;
  p.mt = (c.T + kBM - 1) / kBM;
  p.nt = (c.d + 255) / 256;
  p.kiters = L.Ep / kBK;
  p.hdr = a.hdr;
  p.tabs = a.tabs;
  return launch<RouterDx>(p, s);
}

// In-kernel clock sums: set or clear the switch and zero the sums (on the current device), and
// read them back; both synchronise with the device.
cudaError_t clock_profile_set(bool on) {
  const int v = on ? 1 : 0;
  static const unsigned long long zero[kKCount][2] = {};
  cudaError_t e = cudaMemcpyToSymbol(g_clock_acc, zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_clock_on, &v, sizeof(v));
  return e;
}

cudaError_t clock_profile_read(unsigned long long (*acc)[2]) {
  return cudaMemcpyFromSymbol(acc, g_clock_acc, sizeof(unsigned long long) * 2 * kKCount);
}

}  // namespace moe
