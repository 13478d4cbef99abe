// Internal definitions shared by the layer's translation units: limits, the workspace layout,
// device-side error recording and the bounded-wait clock.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kMaxE = 256;
constexpr int kMaxS = 8;
constexpr int kMaxG = kMaxE + kMaxS;       // routed + shared segments
constexpr int kRowTile = 256;              // CTA-pair GEMM M tile; segments are padded to it
constexpr int kRouterTile = 128;           // tokens per router tensor-core tile
constexpr int kScanChunk = 4096;           // assignments per dispatch-scan block
constexpr int kScanThreads = 512;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s bound on any device wait

// Where a device error was raised (recorded beside the status code).
enum Site : int32_t {
  kSiteScanLookback = 1,
  kSiteScanIndex = 2,
  kSiteGemmProducer = 10,
  kSiteGemmMma = 11,
  kSiteGemmEpilogue = 12,
};

// Header at workspace offset 0.  `status`..`timeout_ns` persist across calls (cleared by
// moe_workspace_init / moe_check_error); the dispatch counters are reset by every dispatch.
struct Hdr {
  int32_t status;
  int32_t site;
  int32_t stall_block_p1;   // test hook: scan block (value - 1) never publishes (0 off)
  int32_t stall_fill_p1;    // test hook: the expert GEMMs' first CTA pair skips fill (value - 1) (0 off)
  uint64_t timeout_ns;      // 0 = kDefaultTimeoutNs
  uint32_t scan_ticket;     // dynamic block index of the dispatch scan
  uint32_t scan_done;       // scan blocks finished; the last one builds the tables
  uint32_t reserved[56];
};
static_assert(sizeof(Hdr) == 256, "header is 256 bytes");
constexpr size_t kHdrResetOffset = offsetof(Hdr, scan_ticket);   // per-dispatch part
constexpr size_t kHdrResetBytes = 8;

// Routing tables written by the last dispatch-scan block.
struct Tables {
  int32_t G;                     // segments = E + S
  int32_t n_mtiles;              // P_G / kRowTile
  int32_t total_rows;            // P_G
  int32_t total_pad;             // pad rows over all segments
  int32_t counts[kMaxE];         // raw demand per routed expert
  int32_t kept[kMaxG];           // rows per segment
  int32_t offsets[kMaxE + 1];    // exact exclusive scan of kept over routed experts
  int32_t poff[kMaxG + 1];       // padded segment starts P_g
  int32_t pad_start[kMaxG + 1];  // exclusive scan of pad rows per segment
  int32_t seg_order[kMaxG];      // segments by padded rows, descending (ties: lower index)
};

// Byte offsets of every workspace region (host computed, passed to kernels as pointers).
struct Layout {
  int64_t rows;          // row capacity of the padded expert-ordered buffers
  int nscan;             // dispatch-scan blocks
  int ntf;               // 128-wide tiles over d_ff
  int ndg;               // per-row gate-gradient partials (two 64-column halves per d_ff tile)
  int nsplit_dwr;        // token splits of dW_r = x^T dlogits (router_dwr_splits)
  int nblk_router;       // router backward blocks (db partials)
  int Ep;                // E rounded up to 64: row length of the bf16 router operands
  size_t hdr, tabs, scan_status, rank, prow_of_slot, slot_of_prow, gate_of_prow, dg_part,
      dlogits, dwr_part, db_part, dgates, xperm, dy_perm, buf_f0, buf_f1, buf_f2, buf_f3, buf_d1,
      dl_bf16, wr_bf16, wr3;
  size_t tok_of_prow;       // token of every padded expert row (pad rows: token 0), for gathered loads
  size_t rt_part, rt_cnt;   // streaming router (E <= 32): partial logits and part counters
  size_t fp8s;              // FP8 backward: row scales of the x, dY and [dA | dB] rows, [3][rows] fp32
  size_t total;
};

struct Cfg {               // validated configuration with derived sizes
  int T, d, f, E, k, S, G, renorm;
  int C;                   // capacity (INT32_MAX when dropless)
  int keep;                // rows with kept a, b: keep_rows rounded down to kRowTile (clamped by the layout)
  int gather_in_gemm;      // fused layer calls: x, dy rows gathered by the GEMMs from token order
};

// ---------------------------------------------------------------------------------------------
// device-side error word and clock
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void record_error(Hdr* h, int32_t code, int32_t site) {
  if (atomicCAS(&h->status, 0, code) == 0) h->site = site;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t wait_limit_ns(const Hdr* h) {
  uint64_t t = *((volatile const uint64_t*)&h->timeout_ns);
  return t ? t : kDefaultTimeoutNs;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Logistic sigmoid 1 / (1 + e^-a) of the SwiGLU epilogues with the approximate reciprocal.  The
// IEEE fp32 division ends in a range check and a branch to a slow path, which keeps the compiler
// from overlapping the elements of a row: with one epilogue warp per SM sub-partition nothing else
// hides that latency.  The approximate reciprocal is within a couple of fp32 ulps, far below the
// bf16 rounding of every output; for a < -88, e^-a overflows to +inf and the reciprocal gives 0,
// the limit.
__device__ __forceinline__ float sigmoid_fast(float a) { return __fdividef(1.f, 1.f + __expf(-a)); }

// ---------------------------------------------------------------------------------------------
// host-side helpers shared by the launchers
// ---------------------------------------------------------------------------------------------

Layout make_layout(const Cfg& c);
// `saved` of the fused layer calls: idx int32 [T,k], gates fp32 [T,k], then (from the 256-byte
// boundary a_off) the kept a and b [keep_rows, d_ff] bf16 one after the other.
struct SavedLayout { size_t logits_off, logits_bytes, a_off, b_off, total; int keep; };
SavedLayout saved_layout(const Cfg& c);
int router_dwr_splits(const Cfg& c);
// tokens of each dW_r split: T / n rounded up to whole 64-token K blocks (the last split is shorter)
inline int router_dwr_ksplit(int T, int n) { return ((T + n - 1) / n + 63) / 64 * 64; }
moe_status_t make_cfg(const moe_config_t* in, Cfg* c);   // validate a configuration
moe_status_t check_device();                     // MOE_OK on an sm_103 device
int num_sms();                                   // SMs of the current device (cached)
moe_status_t cuda_status(cudaError_t e);          // MOE_OK or MOE_ERR_CUDA (clears the error)

// Kernel event profiler (off unless moe_profile_enable(1)): every launch site brackets its kernel
// with prof_mark(id, s, true/false), which records CUDA events on the launching stream.
enum KernelId : int {
  kKRoute = 0, kKScan, kKGather, kKGateUp, kKDown, kKCombine, kKBwdFused, kKWgrad, kKDgradX,
  kKDgates, kKRouterDlogits, kKRouterDwr, kKRouterReduce, kKCombineBwd, kKBwdDh, kKRouterDx, kKSwigluKept,
  kKGateUpFp8, kKQuantE4m3, kKDownFp8, kKQuantCols, kKBwdDhFp8, kKBwdFusedFp8, kKDgradXFp8, kKSplitWr,
  kKToBf16, kKCount
};
void prof_mark(int id, cudaStream_t s, bool begin);
// In-kernel SM clock of the GEMM kernels (gemm.cu): per kernel id, summed clock64 cycles and
// globaltimer nanoseconds of their CTAs while enabled.
cudaError_t clock_profile_set(bool on);
cudaError_t clock_profile_read(unsigned long long (*acc)[2]);

// Launchers implemented in the kernel translation units.  All enqueue on `s` and return the
// launch status.
struct RouteArgs {
  const uint16_t* x; const float* W_r; const float* b_r;
  int32_t* idx; float* gates; float* logits;
};
cudaError_t launch_route(const Cfg& c, const RouteArgs& a, cudaStream_t s);

struct DispatchArgs {
  const int32_t* idx; const uint16_t* x; const uint16_t* dy; const float* gates;
  int32_t* counts; int32_t* offsets; int32_t* row_of_slot; int32_t* token_of_row;
  uint16_t* x_perm; uint16_t* dy_perm;
  Hdr* hdr; Tables* tabs; uint32_t* scan_status; int32_t* rank;
  int32_t* prow_of_slot; int32_t* slot_of_prow; float* gate_of_prow;
  // FP8 forward: per-token row scales carried beside the gathered e4m3 rows (nullable)
  const float* xs_tok; float* xs_perm;
  // nullable: receives the header's status (MOE_OK or the first device error of this dispatch)
  // once the last scan block has built the tables
  int32_t* status_out;
  // nullable: the token of every padded expert row (pad rows: token 0), for GEMMs that gather their
  // operand rows from token order instead of reading x_perm / dY_perm
  int32_t* tok_of_prow;
  // FP8 backward (quant): e4m3 codes [rows, d] and row scales of every padded x and dY row, written
  // beside the bf16 rows (pad rows: zero codes, scale 1)
  uint8_t* x8; uint8_t* dy8; float* x8s; float* dy8s;
};
cudaError_t launch_dispatch_scan(const Cfg& c, const Layout& L, const DispatchArgs& a, cudaStream_t s);
// write_meta: the slot/row tables (and tok_of_prow when given); gather_x / gather_dy: copy the rows;
// gates: the gate of every padded row (implied by gather_dy); quant (with all three): also the
// rows' e4m3 codes and scales (a.x8, a.dy8, a.x8s, a.dy8s)
cudaError_t launch_dispatch_gather(const Cfg& c, const Layout& L, const DispatchArgs& a,
                                   bool write_meta, bool gather_x, bool gather_dy, cudaStream_t s,
                                   bool gates = false, bool quant = false);

struct CombineArgs {
  const uint16_t* o_perm; const float* gates; uint16_t* y;
  const Tables* tabs; const int32_t* prow_of_slot;
};
cudaError_t launch_combine(const Cfg& c, const CombineArgs& a, cudaStream_t s);

// dx = dl W_r^T + the token's expert rows of dx_perm: the router term on the tensor cores (bf16
// operands of E padded to Ep) into r [T, d] bf16, then a token-owner gather adds the rows.
struct RouterDxArgs {
  const uint16_t* dl_bf16; const uint16_t* wr_bf16; uint16_t* r; Hdr* hdr; const Tables* tabs;
};
cudaError_t launch_router_dx(const Cfg& c, const Layout& L, const RouterDxArgs& a, cudaStream_t s);
struct CombineBwdArgs {
  const uint16_t* dx_perm; const uint16_t* r; uint16_t* dx;   // r nullable (no router term)
  const Tables* tabs; const int32_t* prow_of_slot;
};
cudaError_t launch_combine_bwd(const Cfg& c, const CombineBwdArgs& a, cudaStream_t s);

struct RouterBwdArgs {
  const uint16_t* x; const float* W_r; const float* b_r; const int32_t* idx; const float* gates;
  const float* dgates; float* dlogits; float* dW_r; float* db_r;
  float* dwr_part; float* db_part;
};
cudaError_t launch_router_dlogits(const Cfg& c, const Layout& L, const RouterBwdArgs& a, cudaStream_t s);
// the same from the logits the layer forward kept (not read with renormalised gates): dl in fp32,
// the bf16 rows [T, Ep] and router_saved_blocks(c) db partials
cudaError_t launch_router_dlogits_saved(const Cfg& c, const Layout& L, const RouterBwdArgs& a, const float* logits,
                                        uint16_t* dl_bf16, cudaStream_t s);
int router_saved_blocks(const Cfg& c);
// dW_r and db from their partials (nblk db partials)
cudaError_t launch_router_reduce(const Cfg& c, const Layout& L, const RouterBwdArgs& a, int nblk, cudaStream_t s);
// dW_r partials over token splits on the tensor cores (x and the bf16 dlogits, both MN-major)
cudaError_t launch_router_dwr(const Cfg& c, const Layout& L, const uint16_t* x, const uint16_t* dl_bf16,
                              float* dwr_part, Hdr* hdr, const Tables* tabs, cudaStream_t s);
// dst [rows, ld] bf16 = src [rows, cols] fp32, zero for cols <= c < ld
cudaError_t launch_to_bf16_rows(const float* src, int rows, int cols, int ld, uint16_t* dst, cudaStream_t s);

// Router logits on the tensor cores (E <= 128, k <= 8): W_r [d, E] fp32 is split into
// hi + mid + lo bf16 parts stored K-major as wr3 [3][Ep][d].
bool router_on_tensor_cores(const Cfg& c);
bool router_bwd_on_tensor_cores(const Cfg& c);   // the backward too (gates not renormalised)
cudaError_t launch_split_wr(const float* W_r, int d, int E, int Ep, uint16_t* wr3, cudaStream_t s);
struct RouterTcArgs {
  const uint16_t* x; const uint16_t* wr3; const float* b_r;
  int32_t* idx; float* gates; float* logits;                               // forward (read in bwd)
  const float* dgates; float* dlogits; uint16_t* dl_bf16; float* db_part;   // backward
  Hdr* hdr; const Tables* tabs;
};
cudaError_t launch_route_tc(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s);
cudaError_t launch_router_dlogits_tc(const Cfg& c, const Layout& L, const RouterTcArgs& a, cudaStream_t s);

// Router logits for E <= 32 and k <= 8, streaming x once with K split across CTAs
// (route_tc.cu): W_r's three bf16 parts stacked along N in wstack [Nb][d] (written by the launch
// into the workspace's wr3 region), partial logits per (tile, part), counters per token quarter.
struct RouterStreamPlan {
  int eb;          // E rounded up to 8, 16 or 32
  int ntiles;      // 128-token tiles
  int nslice;      // 256-wide K slices
  int nranges;     // CTAs, each a contiguous run of (tile, slice) pairs
  int maxseg;      // the most runs one tile is split between
};
bool router_stream_eligible(const Cfg& c);
RouterStreamPlan router_stream_plan(const Cfg& c);
struct RouterStreamArgs {
  const uint16_t* x; const float* W_r; const float* b_r; uint16_t* wstack; float* part; uint32_t* cnt;
  int32_t* idx; float* gates; float* logits;                            // forward (idx, gates read in bwd)
  const float* dgates; float* dlogits; uint16_t* dl_bf16; float* db_part;   // backward
  Hdr* hdr;
};
cudaError_t launch_route_stream(const Cfg& c, const Layout& L, const RouterStreamArgs& a, cudaStream_t s);
cudaError_t launch_router_dlogits_stream(const Cfg& c, const Layout& L, const RouterStreamArgs& a,
                                         cudaStream_t s);

struct DgatesArgs {
  const float* dg_part; const int32_t* prow_of_slot; float* dgates;
};
cudaError_t launch_dgates(const Cfg& c, const Layout& L, const DgatesArgs& a, cudaStream_t s);

struct FfnFwdArgs {
  const uint16_t* x_perm; const uint16_t* Wg; const uint16_t* Wu; const uint16_t* Wd;
  uint16_t* h; uint16_t* o_perm; Hdr* hdr; const Tables* tabs;
  uint16_t* a_keep; uint16_t* b_keep;   // [rows, d_ff] bf16: a, b of the first c.keep rows
  // gathered A rows (both non-null): x [T, d] in token order and the token of every padded row;
  // x_perm is then not read
  const uint16_t* x_tok; const int32_t* tok;
};
cudaError_t launch_ffn_fwd(const Cfg& c, const Layout& L, const FfnFwdArgs& a, cudaStream_t s);

struct FfnBwdArgs {
  const uint16_t* x_perm; const uint16_t* dy_perm; const float* gate_of_prow;
  const uint16_t* Wg; const uint16_t* Wu; const uint16_t* Wd;
  uint16_t* dh; uint16_t* dA; uint16_t* dB; uint16_t* Hg; float* dg_part; uint16_t* dx_perm;
  uint16_t* dWg; uint16_t* dWu; uint16_t* dWd; Hdr* hdr; const Tables* tabs;
  // kept a, b of rows [0, c.keep) [rows, d_ff] bf16; null: the forward left them in dB and Hg
  const uint16_t* a_kept; const uint16_t* b_kept;
  // gathered rows (all non-null): x and dy [T, d] in token order and the token of every padded row;
  // x_perm and dy_perm are then not read
  const uint16_t* x_tok; const uint16_t* dy_tok; const int32_t* tok;
};
cudaError_t launch_ffn_bwd(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s);
// SwiGLU backward of the kept rows [0, c.keep): a and b from a.a_kept / a.b_kept (or, when null,
// from a.dB / a.Hg where a granular forward kept them), dh' from a.dh; writes dA, dB, Hg and the
// rows' gate partials.
cudaError_t launch_swiglu_bwd_kept(const Cfg& c, const Layout& L, const FfnBwdArgs& a, cudaStream_t s);

// FP8 (e4m3) rows: codes [rows, cols] and one fp32 scale per row (amax / 448), from bf16 rows.
cudaError_t launch_quantize_rows_e4m3(const uint16_t* src, int64_t rows, int cols, uint8_t* codes, float* scales,
                                      cudaStream_t s, const Tables* tabs = nullptr);
// The same for joined rows: row r is src's row r (cols1 values) then src2's row r (cols2 values).
cudaError_t launch_quantize_rows2_e4m3(const uint16_t* src, int cols1, const uint16_t* src2, int cols2, int64_t rows,
                                       uint8_t* codes, float* scales, cudaStream_t s, const Tables* tabs = nullptr);
// FP8 columns: for each of G experts, the source [top (rows_top rows); bottom (rows_bot rows)] x cols
// bf16 gives codes [cols, rows_top + rows_bot] (transposed) and one scale per column.
cudaError_t launch_quantize_cols_e4m3(const uint16_t* top, const uint16_t* bottom, int64_t G, int rows_top,
                                      int rows_bot, int cols, uint8_t* codes, float* scales, cudaStream_t s);
// H = silu(a) * b with a, b from e4m3 rows of x_perm and of W_gate / W_up and their row scales.
struct GateUpFp8Args {
  const uint8_t* x8; const float* xs; const uint8_t* wg8; const float* gs; const uint8_t* wu8;
  const float* us; uint16_t* h; Hdr* hdr; const Tables* tabs;
};
cudaError_t launch_gate_up_fp8(const Cfg& c, const Layout& L, const GateUpFp8Args& a, cudaStream_t s);
// The FP8 backward of the expert FFN: e4m3 codes of the x and dY rows (per row), the forward's
// weight codes (recompute), W_d's columns [G, f, d] (one scale per d_ff channel) and the joined
// columns of W_gate and W_up [G, d, 2f] (one scale per d_model channel); bf16 dh', dA, dB, Hg,
// the joined [dA | dB] rows' codes and scales, dx_perm and the weight gradients.
struct FfnBwd8Args {
  const uint16_t* x_perm; const uint16_t* dy_perm;
  const uint8_t* x8; const float* xs; const uint8_t* dy8; const float* dys;
  const uint8_t* wg8; const float* gs; const uint8_t* wu8; const float* us;
  const uint8_t* wdt8; const float* wdts; const uint8_t* wgut8; const float* wguts;
  const float* gate_of_prow;
  uint16_t* dh; uint16_t* dA; uint16_t* dB; uint16_t* Hg; float* dg_part;
  uint8_t* dab8; float* dabs; uint16_t* dx_perm;
  uint16_t* dWg; uint16_t* dWu; uint16_t* dWd; Hdr* hdr; const Tables* tabs;
};
cudaError_t launch_ffn_bwd_fp8(const Cfg& c, const Layout& L, const FfnBwd8Args& a, cudaStream_t s);
// O = H W_d^T from e4m3 rows of H and of W_d (one scale per output channel).
struct DownFp8Args {
  const uint8_t* h8; const float* hs; const uint8_t* wd8; const float* ds; uint16_t* o; Hdr* hdr;
  const Tables* tabs;
};
cudaError_t launch_down_fp8(const Cfg& c, const Layout& L, const DownFp8Args& a, cudaStream_t s);

}  // namespace moe
