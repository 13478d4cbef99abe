// The C ABI (include/moe.h): argument validation, workspace layout and the composition of the
// layer's forward and backward from the kernels of route.cu, dispatch.cu, gemm.cu and combine.cu.
#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace moe {

int route_block_tokens(int E);   // route.cu

namespace {

constexpr size_t kAlign = 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

moe_status_t make_cfg(const moe_config_t* in, Cfg* c) {
  if (in == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_config_t& m = *in;
  if (m.T < 1 || m.T > (1 << 20) || m.E < 1 || m.E > kMaxE || m.k < 1 || m.k > m.E ||
      m.n_shared < 0 || m.n_shared > kMaxS || m.d_model < 64 || m.d_ff < 64 ||
      m.d_model > 16384 || m.d_ff > 16384 || (m.d_model % 64) != 0 || (m.d_ff % 64) != 0 ||
      (int64_t)m.T * m.k > (int64_t)1 << 24 || !(m.capacity_factor == m.capacity_factor) || m.keep_rows < 0 ||
      (m.gather_in_gemm != 0 && m.gather_in_gemm != 1))
    return MOE_ERR_INVALID_ARG;
  c->T = m.T;
  c->d = m.d_model;
  c->f = m.d_ff;
  c->E = m.E;
  c->k = m.k;
  c->S = m.n_shared;
  c->G = m.E + m.n_shared;
  c->renorm = m.renorm ? 1 : 0;
  c->keep = m.keep_rows / kRowTile * kRowTile;   // clamped to the row capacity by make_layout users
  c->gather_in_gemm = m.gather_in_gemm;
  if (m.capacity_factor > 0.f) {
    const double cap = std::ceil((double)m.capacity_factor * (double)m.T * (double)m.k / (double)m.E);
    c->C = cap >= (double)INT_MAX ? INT_MAX : (int)cap;
  } else {
    c->C = INT_MAX;
  }
  return MOE_OK;
}

moe_status_t check_device() {
  static int ok = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      ok = 0;
      return;
    }
    ok = (major == 10 && minor == 3) ? 1 : 0;
  });
  return ok == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

namespace {

struct Ws {
  Layout L;
  char* base;
  Hdr* hdr() const { return reinterpret_cast<Hdr*>(base + L.hdr); }
  Tables* tabs() const { return reinterpret_cast<Tables*>(base + L.tabs); }
  template <class T> T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

moe_status_t get_ws(const Cfg& c, void* ws, size_t ws_bytes, Ws* w) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  w->L = make_layout(c);
  if (ws_bytes < w->L.total) return MOE_ERR_WORKSPACE;
  w->base = static_cast<char*>(ws);
  return MOE_OK;
}

DispatchArgs dispatch_args(const Ws& w) {
  DispatchArgs a{};
  a.hdr = w.hdr();
  a.tabs = w.tabs();
  a.scan_status = w.at<uint32_t>(w.L.scan_status);
  a.rank = w.at<int32_t>(w.L.rank);
  a.prow_of_slot = w.at<int32_t>(w.L.prow_of_slot);
  a.slot_of_prow = w.at<int32_t>(w.L.slot_of_prow);
  a.gate_of_prow = w.at<float>(w.L.gate_of_prow);
  return a;
}

}  // namespace

// Token splits of the dW_r product (x^T dl, one read of x): the persistent kernel deals its
// (d_model tile, split) jobs round-robin to 152 CTAs, so take the split count whose busiest CTA
// streams the fewest tokens (plus a small fixed cost a job), among counts whose fp32 partials
// (splits x d_model x E x 4 bytes) stay within about a fifth of x.  Fixed by the configuration, not the
// device, so the order of the fixed-order sum of the partials is too.
int router_dwr_splits(const Cfg& c) {
  constexpr int kCtas = 152;
  constexpr long long kJobCost = 32;   // tokens' worth of fixed cost per job
  const int mt = (c.d + 127) / 128;
  const int nmax = std::max(1, std::min(c.T / (10 * c.E), 256));
  int best = 1;
  long long best_cost = -1;
  for (int n = 1; n <= nmax; ++n) {
    const long long waves = ((long long)mt * n + kCtas - 1) / kCtas;
    const long long cost = waves * (router_dwr_ksplit(c.T, n) + kJobCost);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = n;
    }
  }
  return best;
}

Layout make_layout(const Cfg& c) {
  Layout L{};
  const int64_t routed = ((int64_t)c.T * c.k + (int64_t)(kRowTile - 1) * c.E + kRowTile - 1) / kRowTile * kRowTile;
  const int64_t shared = (int64_t)c.S * (((int64_t)c.T + kRowTile - 1) / kRowTile * kRowTile);
  L.rows = routed + shared;
  L.nscan = (int)(((int64_t)c.T * c.k + kScanChunk - 1) / kScanChunk);
  L.ntf = (c.f + 127) / 128;
  L.ndg = 2 * L.ntf;
  // db partials: one per 32 tokens from the tensor-core backward, else one per SIMT router block
  L.nblk_router = router_bwd_on_tensor_cores(c) ? 4 * ((c.T + kRouterTile - 1) / kRouterTile)
                                                : (c.T + route_block_tokens(c.E) - 1) / route_block_tokens(c.E);
  L.nsplit_dwr = router_dwr_splits(c);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const size_t rows = (size_t)L.rows;
  L.hdr = take(sizeof(Hdr));
  L.tabs = take(sizeof(Tables));
  L.scan_status = take((size_t)L.nscan * c.E * 4);
  L.rank = take((size_t)c.T * c.k * 4);
  L.prow_of_slot = take((size_t)c.T * c.k * 4);
  L.slot_of_prow = take(rows * 4);
  L.gate_of_prow = take(rows * 4);
  L.dg_part = take(rows * L.ndg * 4);
  L.dlogits = take((size_t)c.T * c.E * 4);
  L.dwr_part = take((size_t)L.nsplit_dwr * c.d * c.E * 4);
  L.db_part = take((size_t)std::max(L.nblk_router, router_saved_blocks(c)) * c.E * 4);
  L.dgates = take((size_t)c.T * c.k * 4);
  L.xperm = take(rows * c.d * 2);
  L.dy_perm = take(rows * c.d * 2);
  L.buf_f0 = take(rows * c.f * 2);
  L.buf_f1 = take(rows * c.f * 2);
  L.buf_f2 = take(rows * c.f * 2);
  L.buf_f3 = take(rows * c.f * 2);
  L.buf_d1 = take(rows * c.d * 2);
  L.Ep = (c.E + 63) / 64 * 64;
  L.dl_bf16 = take((size_t)c.T * L.Ep * 2);
  L.wr_bf16 = take((size_t)c.d * L.Ep * 2);
  L.wr3 = take((size_t)3 * L.Ep * c.d * 2);
  L.fp8s = take(rows * 3 * 4);
  L.tok_of_prow = take(rows * 4);
  if (router_stream_eligible(c)) {
    const RouterStreamPlan pl = router_stream_plan(c);
    L.rt_part = take(pl.maxseg > 1 ? (size_t)pl.ntiles * pl.maxseg * pl.eb * 128 * 4 : 0);
    L.rt_cnt = take((size_t)pl.ntiles * 4 * 4);
  }
  L.total = off;
  return L;
}

// idx [T, k], gates [T, k]; the logits [T, E] fp32 when the gates are not renormalised (the
// router backward's softmax reads them instead of a second pass over x); the kept a and b.
SavedLayout saved_layout(const Cfg& c) {
  SavedLayout sl{};
  sl.keep = (int)std::min<int64_t>(c.keep, make_layout(c).rows);
  size_t off = (size_t)c.T * c.k * 8;
  sl.logits_bytes = c.renorm ? 0 : (size_t)c.T * c.E * 4;
  if (sl.logits_bytes != 0) {
    sl.logits_off = align_up(off, 256);
    off = sl.logits_off + sl.logits_bytes;
  }
  const size_t kept = (size_t)sl.keep * c.f * 2;
  if (sl.keep == 0) {
    sl.a_off = sl.b_off = sl.total = off;
    return sl;
  }
  sl.a_off = align_up(off, 256);
  sl.b_off = sl.a_off + kept;
  sl.total = sl.b_off + kept;
  return sl;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 148;
  }
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      n = 148;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

moe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  (void)cudaGetLastError();
  return MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------------
// kernel event profiler
// ---------------------------------------------------------------------------------------------

namespace {

const char* const kKernelNames[] = {
    "route_fwd", "dispatch_scan", "dispatch_gather", "gemm_gate_up_swiglu", "gemm_down",
    "combine", "gemm_bwd_recompute_swiglu", "gemm_wgrad", "gemm_dgrad_x", "dgates_reduce",
    "router_dlogits", "router_dwr", "router_reduce", "combine_bwd", "gemm_bwd_dgrad_down",
    "gemm_router_dx", "swiglu_bwd_kept", "gemm_gate_up_fp8", "quantize_e4m3", "gemm_down_fp8",
    "quantize_cols_e4m3", "gemm_bwd_dgrad_down_fp8", "gemm_bwd_recompute_swiglu_fp8", "gemm_dgrad_x_fp8",
    "router_split_wr", "to_bf16_rows"};
static_assert(sizeof(kKernelNames) / sizeof(kKernelNames[0]) == kKCount, "a name for every kernel id");

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;           // events, reused across enables
  size_t used = 0;
  std::vector<std::pair<int, std::pair<size_t, size_t>>> marks;   // (kernel, (start, stop))
  size_t open[kKCount];
  double total_ms[kKCount];
  int launches[kKCount];
};

Profiler& profiler() {
  static Profiler p;
  return p;
}

}  // namespace

void prof_mark(int id, cudaStream_t s, bool begin) {
  Profiler& p = profiler();
  if (!p.on) return;
  std::lock_guard<std::mutex> lock(p.mu);
  if (p.used == p.pool.size()) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) {
      (void)cudaGetLastError();
      return;
    }
    p.pool.push_back(ev);
  }
  const size_t e = p.used++;
  if (cudaEventRecord(p.pool[e], s) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  if (begin) {
    p.open[id] = e;
  } else {
    p.marks.push_back({id, {p.open[id], e}});
  }
}

}  // namespace moe

using namespace moe;

#define MOE_TRY(expr)                         \
  do {                                        \
    const moe_status_t _st = (expr);          \
    if (_st != MOE_OK) return _st;            \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))
#define MOE_NEED(cond) \
  do {                 \
    if (!(cond)) return MOE_ERR_INVALID_ARG; \
  } while (0)

namespace {

moe_status_t do_dispatch(const Cfg& c, const Ws& w, const int32_t* idx, const uint16_t* x,
                         const uint16_t* dy, const float* gates, int32_t* counts, int32_t* offsets,
                         int32_t* row_of_slot, int32_t* token_of_row, uint16_t* x_perm,
                         uint16_t* dy_perm, cudaStream_t s) {
  DispatchArgs a = dispatch_args(w);
  a.idx = idx;
  a.x = x;
  a.dy = dy;
  a.gates = gates;
  a.counts = counts;
  a.offsets = offsets;
  a.row_of_slot = row_of_slot;
  a.token_of_row = token_of_row;
  a.x_perm = x_perm;
  a.dy_perm = dy_perm;
  MOE_CUDA(launch_dispatch_scan(c, w.L, a, s));
  MOE_CUDA(launch_dispatch_gather(c, w.L, a, true, true, dy != nullptr, s));
  return MOE_OK;
}

// The dispatch of the fused calls: the queues and tables only, the token of every padded row (the
// expert GEMMs gather their rows from token order), and for the backward the gate of every row.
moe_status_t do_dispatch_tables(const Cfg& c, const Ws& w, const int32_t* idx, const float* gates, cudaStream_t s) {
  DispatchArgs a = dispatch_args(w);
  a.idx = idx;
  a.gates = gates;
  a.tok_of_prow = w.at<int32_t>(w.L.tok_of_prow);
  MOE_CUDA(launch_dispatch_scan(c, w.L, a, s));
  MOE_CUDA(launch_dispatch_gather(c, w.L, a, true, false, false, s, gates != nullptr));
  return MOE_OK;
}

// x_perm / dy_perm, or (tok non-null) x and dy in token order with the token of every padded row.
moe_status_t do_ffn_bwd(const Cfg& c, const Ws& w, const uint16_t* x_perm, const uint16_t* dy_perm,
                        const uint16_t* Wg, const uint16_t* Wu, const uint16_t* Wd,
                        uint16_t* dx_perm, float* dgates, uint16_t* dWg, uint16_t* dWu,
                        uint16_t* dWd, const uint16_t* a_kept, const uint16_t* b_kept, cudaStream_t s,
                        const uint16_t* x_tok = nullptr, const uint16_t* dy_tok = nullptr,
                        const int32_t* tok = nullptr) {
  FfnBwdArgs b{};
  b.x_tok = x_tok;
  b.dy_tok = dy_tok;
  b.tok = tok;
  b.x_perm = x_perm;
  b.dy_perm = dy_perm;
  b.gate_of_prow = w.at<float>(w.L.gate_of_prow);
  b.Wg = Wg;
  b.Wu = Wu;
  b.Wd = Wd;
  b.dh = w.at<uint16_t>(w.L.buf_f3);
  b.dA = w.at<uint16_t>(w.L.buf_f0);
  b.dB = w.at<uint16_t>(w.L.buf_f1);   // granular calls: holds the kept a of rows [0, c.keep)
  b.Hg = w.at<uint16_t>(w.L.buf_f2);   // granular calls: holds the kept b likewise
  b.a_kept = a_kept;                    // fused calls: the kept a and b in `saved`
  b.b_kept = b_kept;
  b.dg_part = w.at<float>(w.L.dg_part);
  b.dx_perm = dx_perm;
  b.dWg = dWg;
  b.dWu = dWu;
  b.dWd = dWd;
  b.hdr = w.hdr();
  b.tabs = w.tabs();
  MOE_CUDA(launch_ffn_bwd(c, w.L, b, s));
  DgatesArgs g{};
  g.dg_part = b.dg_part;
  g.prow_of_slot = w.at<int32_t>(w.L.prow_of_slot);
  g.dgates = dgates;
  MOE_CUDA(launch_dgates(c, w.L, g, s));
  return MOE_OK;
}

// The FP8 expert-FFN backward on the rows moe_dispatch laid out (x_perm, dy_perm, gates per row).
// Scratch: the x and dY rows' codes share buf_d1 (free until dgrad x writes dx_perm there), their
// scales and the [dA | dB] rows' scales go to fp8s, the [dA | dB] codes to buf_f3 once dh' is used.
// The FP8 backward's dispatch: the queues from the saved idx, the bf16 x and dY rows (the weight
// gradients' operands) and, from the same pass over each token's rows, their e4m3 codes and row
// scales (the dh' and recompute GEMMs' operands): into O/dX's buffer and the FP8 scale planes.
moe_status_t do_dispatch_fp8_bwd(const Cfg& c, const Ws& w, const int32_t* idx, const uint16_t* x,
                                 const uint16_t* dy, const float* gates, cudaStream_t s) {
  const size_t rows = (size_t)w.L.rows;
  DispatchArgs a = dispatch_args(w);
  a.idx = idx;
  a.x = x;
  a.dy = dy;
  a.gates = gates;
  a.x_perm = w.at<uint16_t>(w.L.xperm);
  a.dy_perm = w.at<uint16_t>(w.L.dy_perm);
  a.x8 = w.at<uint8_t>(w.L.buf_d1);
  a.dy8 = a.x8 + rows * c.d;
  a.x8s = w.at<float>(w.L.fp8s);
  a.dy8s = a.x8s + rows;
  MOE_CUDA(launch_dispatch_scan(c, w.L, a, s));
  MOE_CUDA(launch_dispatch_gather(c, w.L, a, true, true, true, s, false, true));
  return MOE_OK;
}

moe_status_t do_ffn_bwd_fp8(const Cfg& c, const Ws& w, const uint8_t* wg8, const float* wg_scale,
                            const uint8_t* wu8, const float* wu_scale, const uint8_t* wdt8,
                            const float* wdt_scale, const uint8_t* wgut8, const float* wgut_scale,
                            float* dgates, uint16_t* dWg, uint16_t* dWu, uint16_t* dWd, cudaStream_t s) {
  // the x and dY rows' codes and scales were written by the dispatch (do_dispatch_fp8_bwd)
  const size_t rows = (size_t)w.L.rows;
  FfnBwd8Args b{};
  b.x_perm = w.at<uint16_t>(w.L.xperm);
  b.dy_perm = w.at<uint16_t>(w.L.dy_perm);
  uint8_t* x8 = w.at<uint8_t>(w.L.buf_d1);
  uint8_t* dy8 = x8 + rows * c.d;
  float* sc = w.at<float>(w.L.fp8s);
  b.x8 = x8;
  b.xs = sc;
  b.dy8 = dy8;
  b.dys = sc + rows;
  b.wg8 = wg8;
  b.gs = wg_scale;
  b.wu8 = wu8;
  b.us = wu_scale;
  b.wdt8 = wdt8;
  b.wdts = wdt_scale;
  b.wgut8 = wgut8;
  b.wguts = wgut_scale;
  b.gate_of_prow = w.at<float>(w.L.gate_of_prow);
  b.dh = w.at<uint16_t>(w.L.buf_f3);
  b.dA = w.at<uint16_t>(w.L.buf_f0);
  b.dB = w.at<uint16_t>(w.L.buf_f1);
  b.Hg = w.at<uint16_t>(w.L.buf_f2);
  b.dg_part = w.at<float>(w.L.dg_part);
  b.dab8 = w.at<uint8_t>(w.L.buf_f3);
  b.dabs = sc + 2 * rows;
  b.dx_perm = w.at<uint16_t>(w.L.buf_d1);
  b.dWg = dWg;
  b.dWu = dWu;
  b.dWd = dWd;
  b.hdr = w.hdr();
  b.tabs = w.tabs();
  MOE_CUDA(launch_ffn_bwd_fp8(c, w.L, b, s));
  DgatesArgs g{};
  g.dg_part = b.dg_part;
  g.prow_of_slot = w.at<int32_t>(w.L.prow_of_slot);
  g.dgates = dgates;
  MOE_CUDA(launch_dgates(c, w.L, g, s));
  return MOE_OK;
}

moe_status_t do_router_bwd(const Cfg& c, const Ws& w, const uint16_t* x, const float* W_r,
                           const float* b_r, const int32_t* idx, const float* gates,
                           const float* dgates, float* dlogits, float* dW_r, float* db_r,
                           cudaStream_t s) {
  RouterBwdArgs a{};
  a.x = x;
  a.W_r = W_r;
  a.b_r = b_r;
  a.idx = idx;
  a.gates = gates;
  a.dgates = dgates;
  a.dlogits = dlogits;
  a.dW_r = dW_r;
  a.db_r = db_r;
  a.dwr_part = w.at<float>(w.L.dwr_part);
  a.db_part = w.at<float>(w.L.db_part);
  uint16_t* dl_bf16 = w.at<uint16_t>(w.L.dl_bf16);
  if (router_bwd_on_tensor_cores(c) && router_stream_eligible(c)) {   // narrow router, x streamed once
    RouterStreamArgs t{x, W_r, b_r, w.at<uint16_t>(w.L.wr3), w.at<float>(w.L.rt_part), w.at<uint32_t>(w.L.rt_cnt),
                       const_cast<int32_t*>(idx), const_cast<float*>(gates), nullptr,
                       dgates, dlogits, dl_bf16, a.db_part, w.hdr()};
    MOE_CUDA(launch_router_dlogits_stream(c, w.L, t, s));
  } else if (router_bwd_on_tensor_cores(c)) {   // logits recomputed on the tensor cores; dl in both types
    uint16_t* wr3 = w.at<uint16_t>(w.L.wr3);
    MOE_CUDA(launch_split_wr(W_r, c.d, c.E, w.L.Ep, wr3, s));
    RouterTcArgs t{x, wr3, b_r, const_cast<int32_t*>(idx), const_cast<float*>(gates), nullptr,
                   dgates, dlogits, dl_bf16, a.db_part, w.hdr(), w.tabs()};
    MOE_CUDA(launch_router_dlogits_tc(c, w.L, t, s));
  } else {
    MOE_CUDA(launch_router_dlogits(c, w.L, a, s));
    MOE_CUDA(launch_to_bf16_rows(dlogits, c.T, c.E, w.L.Ep, dl_bf16, s));
  }
  MOE_CUDA(launch_router_dwr(c, w.L, x, dl_bf16, a.dwr_part, w.hdr(), w.tabs(), s));
  MOE_CUDA(launch_router_reduce(c, w.L, a, w.L.nblk_router, s));
  return MOE_OK;
}

// The layer backward's router gradient: dl from the logits the forward kept in `saved` (the
// softmax needs them only when the gates are not renormalised), so x is read once here, by the
// dW_r product, instead of twice.  Leaves dl's bf16 rows in the workspace for the dx term.
moe_status_t do_router_bwd_saved(const Cfg& c, const Ws& w, const uint16_t* x, const float* logits,
                                 const int32_t* idx, const float* gates, const float* dgates, float* dlogits,
                                 float* dW_r, float* db_r, cudaStream_t s) {
  RouterBwdArgs a{};
  a.x = x;
  a.idx = idx;
  a.gates = gates;
  a.dgates = dgates;
  a.dlogits = dlogits;
  a.dW_r = dW_r;
  a.db_r = db_r;
  a.dwr_part = w.at<float>(w.L.dwr_part);
  a.db_part = w.at<float>(w.L.db_part);
  uint16_t* dl_bf16 = w.at<uint16_t>(w.L.dl_bf16);
  MOE_CUDA(launch_router_dlogits_saved(c, w.L, a, logits, dl_bf16, s));
  MOE_CUDA(launch_router_dwr(c, w.L, x, dl_bf16, a.dwr_part, w.hdr(), w.tabs(), s));
  MOE_CUDA(launch_router_reduce(c, w.L, a, router_saved_blocks(c), s));
  return MOE_OK;
}

// Router forward: narrow routers (E <= 32, k <= 8) stream x once with K split across CTAs; up to
// 128 experts the logits run on the tensor cores one 128-token tile per CTA; else the fp32 tile
// product.  The tensor-core paths split W_r into bf16 parts first.
moe_status_t do_route(const Cfg& c, const Ws& w, const uint16_t* x, const float* W_r, const float* b_r,
                      int32_t* idx, float* gates, float* logits, cudaStream_t s) {
  if (router_stream_eligible(c)) {
    RouterStreamArgs t{x, W_r, b_r, w.at<uint16_t>(w.L.wr3), w.at<float>(w.L.rt_part), w.at<uint32_t>(w.L.rt_cnt),
                       idx, gates, logits, nullptr, nullptr, nullptr, nullptr, w.hdr()};
    MOE_CUDA(launch_route_stream(c, w.L, t, s));
  } else if (router_on_tensor_cores(c)) {
    uint16_t* wr3 = w.at<uint16_t>(w.L.wr3);
    MOE_CUDA(launch_split_wr(W_r, c.d, c.E, w.L.Ep, wr3, s));
    RouterTcArgs t{x, wr3, b_r, idx, gates, logits, nullptr, nullptr, nullptr, nullptr, w.hdr(), w.tabs()};
    MOE_CUDA(launch_route_tc(c, w.L, t, s));
  } else {
    RouteArgs a{x, W_r, b_r, idx, gates, logits};
    MOE_CUDA(launch_route(c, a, s));
  }
  return MOE_OK;
}

// dx = dlogits W_r^T (when dlogits is given) + the token's expert rows of dx_perm.  The router
// term runs on the tensor cores (bf16 copies of dlogits and W_r padded to Ep columns) into a bf16
// [T, d] buffer in the workspace's dY_perm region, which the backward no longer needs here; the
// token-owner gather then adds it to the rows in fp32 with one rounding.
// dl_ready: the workspace already holds dl's bf16 rows (the layer backward's router gradient).
moe_status_t do_combine_bwd(const Cfg& c, const Ws& w, const uint16_t* dx_perm, const float* dlogits,
                            const float* W_r, uint16_t* dx, cudaStream_t s, bool dl_ready = false) {
  uint16_t* r = nullptr;
  if (dlogits != nullptr) {
    uint16_t* dl_bf16 = w.at<uint16_t>(w.L.dl_bf16);
    uint16_t* wr_bf16 = w.at<uint16_t>(w.L.wr_bf16);
    r = w.at<uint16_t>(w.L.dy_perm);
    if (!dl_ready) MOE_CUDA(launch_to_bf16_rows(dlogits, c.T, c.E, w.L.Ep, dl_bf16, s));
    MOE_CUDA(launch_to_bf16_rows(W_r, c.d, c.E, w.L.Ep, wr_bf16, s));
    RouterDxArgs ra{dl_bf16, wr_bf16, r, w.hdr(), w.tabs()};
    MOE_CUDA(launch_router_dx(c, w.L, ra, s));
  }
  CombineBwdArgs a{dx_perm, r, dx, w.tabs(), w.at<int32_t>(w.L.prow_of_slot)};
  MOE_CUDA(launch_combine_bwd(c, a, s));
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_INDEX: return "expert index out of range";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* ws_bytes, size_t* saved_bytes) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(ws_bytes != nullptr);
  *ws_bytes = make_layout(c).total;
  if (saved_bytes) *saved_bytes = saved_layout(c).total;
  return MOE_OK;
}

moe_status_t moe_saved_layout(const moe_config_t* cfg, size_t* logits_off, size_t* logits_bytes, size_t* kept_off,
                              size_t* kept_bytes) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  const SavedLayout sl = saved_layout(c);
  if (logits_off) *logits_off = sl.logits_off;
  if (logits_bytes) *logits_bytes = sl.logits_bytes;
  if (kept_off) *kept_off = sl.a_off;
  if (kept_bytes) *kept_bytes = sl.total - sl.a_off;
  return MOE_OK;
}

// Kept-row count for a byte budget: a and b of one expert-ordered row take 4 d_ff bytes of
// `saved`; rows go in pair-tile multiples (256) up to the row capacity.
moe_status_t moe_keep_rows_for_budget(const moe_config_t* cfg, uint64_t budget_bytes, int32_t* keep_rows,
                                      uint64_t* kept_bytes) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(keep_rows != nullptr);
  const uint64_t per_row = (uint64_t)c.f * 4;
  const int64_t cap = make_layout(c).rows;
  const int64_t rows = std::min<int64_t>((int64_t)(budget_bytes / per_row) / kRowTile * kRowTile, cap);
  *keep_rows = (int32_t)rows;
  if (kept_bytes) *kept_bytes = (uint64_t)rows * per_row;
  return MOE_OK;
}

moe_status_t moe_keep_rows_for_free_memory(const moe_config_t* cfg, uint64_t reserve_bytes, int32_t* keep_rows,
                                           uint64_t* kept_bytes) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(keep_rows != nullptr);
  size_t free_b = 0, total_b = 0;
  MOE_CUDA(cudaMemGetInfo(&free_b, &total_b));
  const uint64_t budget = free_b > reserve_bytes ? (uint64_t)free_b - reserve_bytes : 0;
  return moe_keep_rows_for_budget(cfg, budget, keep_rows, kept_bytes);
}

moe_status_t moe_perm_rows(const moe_config_t* cfg, int64_t* rows) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(rows != nullptr);
  *rows = make_layout(c).rows;
  return MOE_OK;
}

moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_CUDA(cudaMemsetAsync(w.hdr(), 0, sizeof(Hdr), stream));
  return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                       int32_t* idx, float* gates, float* logits, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x && W_r && idx && gates && aligned16(x) && aligned16(W_r) && aligned16(idx) &&
           aligned16(gates) && (!b_r || aligned16(b_r)) && (!logits || aligned16(logits)));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  return do_route(c, w, x, W_r, b_r, idx, gates, logits, stream);
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const int32_t* idx, const moe_bf16* x,
                          int32_t* counts, int32_t* offsets, int32_t* row_of_slot, int32_t* token_of_row,
                          moe_bf16* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(idx && x && counts && offsets && row_of_slot && token_of_row && x_perm);
  MOE_NEED(aligned16(idx) && aligned16(x) && aligned16(counts) && aligned16(offsets) &&
           aligned16(row_of_slot) && aligned16(token_of_row) && aligned16(x_perm));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  return do_dispatch(c, w, idx, x, nullptr, nullptr, counts, offsets, row_of_slot, token_of_row,
                     x_perm, nullptr, stream);
}

moe_status_t moe_expert_ffn_fwd(const moe_config_t* cfg, const moe_bf16* x_perm,
                                const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                                moe_bf16* o_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x_perm && W_gate && W_up && W_down && o_perm);
  MOE_NEED(aligned16(x_perm) && aligned16(W_gate) && aligned16(W_up) && aligned16(W_down) && aligned16(o_perm));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  FfnFwdArgs a{x_perm, W_gate, W_up, W_down, w.at<uint16_t>(w.L.buf_f0), o_perm, w.hdr(), w.tabs(),
               w.at<uint16_t>(w.L.buf_f1), w.at<uint16_t>(w.L.buf_f2)};
  MOE_CUDA(launch_ffn_fwd(c, w.L, a, stream));
  return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* cfg, const moe_bf16* o_perm, const float* gates,
                         moe_bf16* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(o_perm && gates && y && aligned16(o_perm) && aligned16(gates) && aligned16(y));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  CombineArgs a{o_perm, gates, y, w.tabs(), w.at<int32_t>(w.L.prow_of_slot)};
  MOE_CUDA(launch_combine(c, a, stream));
  return MOE_OK;
}

moe_status_t moe_expert_ffn_bwd(const moe_config_t* cfg, const moe_bf16* x_perm, const moe_bf16* dy,
                                const float* gates,
                                const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                                moe_bf16* dx_perm, float* dgates,
                                moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x_perm && dy && gates && W_gate && W_up && W_down && dx_perm && dgates && dW_gate &&
           dW_up && dW_down);
  MOE_NEED(aligned16(x_perm) && aligned16(dy) && aligned16(gates) && aligned16(W_gate) &&
           aligned16(W_up) && aligned16(W_down) && aligned16(dx_perm) && aligned16(dgates) &&
           aligned16(dW_gate) && aligned16(dW_up) && aligned16(dW_down));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  DispatchArgs a = dispatch_args(w);
  a.dy = dy;
  a.gates = gates;
  a.dy_perm = w.at<uint16_t>(w.L.dy_perm);
  MOE_CUDA(launch_dispatch_gather(c, w.L, a, false, false, true, stream));
  return do_ffn_bwd(c, w, x_perm, a.dy_perm, W_gate, W_up, W_down, dx_perm, dgates, dW_gate, dW_up,
                    dW_down, nullptr, nullptr, stream);
}

moe_status_t moe_router_bwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                            const int32_t* idx, const float* gates, const float* dgates,
                            float* dlogits, float* dW_r, float* db_r,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x && W_r && idx && gates && dgates && dlogits && dW_r);
  MOE_NEED(aligned16(x) && aligned16(W_r) && aligned16(idx) && aligned16(gates) && aligned16(dgates) &&
           aligned16(dlogits) && aligned16(dW_r) && (!b_r || aligned16(b_r)) && (!db_r || aligned16(db_r)));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  return do_router_bwd(c, w, x, W_r, b_r, idx, gates, dgates, dlogits, dW_r, db_r, stream);
}

moe_status_t moe_combine_bwd(const moe_config_t* cfg, const moe_bf16* dx_perm, const float* dlogits,
                             const float* W_r, moe_bf16* dx, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(dx_perm && dx && aligned16(dx_perm) && aligned16(dx));
  MOE_NEED(!dlogits || (W_r && aligned16(dlogits) && aligned16(W_r)));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  return do_combine_bwd(c, w, dx_perm, dlogits, W_r, dx, stream);
}

moe_status_t moe_quantize_rows_e4m3(const moe_bf16* src, int64_t rows, int32_t cols, uint8_t* codes,
                                    float* scales, moe_stream_t stream) {
  MOE_NEED(rows >= 0 && cols > 0 && cols % 16 == 0 && cols <= 16384 && rows <= ((int64_t)1 << 31));
  MOE_NEED(rows == 0 || (src && codes && scales && aligned16(src) && aligned16(codes) && aligned16(scales)));
  MOE_TRY(check_device());
  MOE_CUDA(launch_quantize_rows_e4m3(src, rows, cols, codes, scales, stream));
  return MOE_OK;
}

moe_status_t moe_gate_up_fp8(const moe_config_t* cfg, const uint8_t* x8, const float* x_scale, const uint8_t* wg8,
                             const float* wg_scale, const uint8_t* wu8, const float* wu_scale, moe_bf16* h,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x8 && x_scale && wg8 && wg_scale && wu8 && wu_scale && h);
  MOE_NEED(aligned16(x8) && aligned16(x_scale) && aligned16(wg8) && aligned16(wg_scale) && aligned16(wu8) &&
           aligned16(wu_scale) && aligned16(h));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  GateUpFp8Args a{x8, x_scale, wg8, wg_scale, wu8, wu_scale, h, w.hdr(), w.tabs()};
  MOE_CUDA(launch_gate_up_fp8(c, w.L, a, stream));
  return MOE_OK;
}

moe_status_t moe_down_fp8(const moe_config_t* cfg, const uint8_t* h8, const float* h_scale, const uint8_t* wd8,
                          const float* wd_scale, moe_bf16* o_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(h8 && h_scale && wd8 && wd_scale && o_perm);
  MOE_NEED(aligned16(h8) && aligned16(h_scale) && aligned16(wd8) && aligned16(wd_scale) && aligned16(o_perm));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  DownFp8Args a{h8, h_scale, wd8, wd_scale, o_perm, w.hdr(), w.tabs()};
  MOE_CUDA(launch_down_fp8(c, w.L, a, stream));
  return MOE_OK;
}

moe_status_t moe_layer_fwd_fp8(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                               const uint8_t* wg8, const float* wg_scale, const uint8_t* wu8,
                               const float* wu_scale, const uint8_t* wd8, const float* wd_scale, moe_bf16* y,
                               void* saved, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  // its scratch lives in the backward's buffers, where kept activations would have to survive
  MOE_NEED(cfg->keep_rows == 0);
  MOE_NEED(x && W_r && wg8 && wg_scale && wu8 && wu_scale && wd8 && wd_scale && y && saved);
  MOE_NEED(aligned16(x) && aligned16(W_r) && (!b_r || aligned16(b_r)) && aligned16(wg8) && aligned16(wg_scale) &&
           aligned16(wu8) && aligned16(wu_scale) && aligned16(wd8) && aligned16(wd_scale) && aligned16(y) &&
           aligned16(saved));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  int32_t* idx = static_cast<int32_t*>(saved);
  float* gates = reinterpret_cast<float*>(idx + (size_t)c.T * c.k);
  const SavedLayout sv = saved_layout(c);
  float* logits = sv.logits_bytes ? reinterpret_cast<float*>(static_cast<char*>(saved) + sv.logits_off) : nullptr;
  MOE_TRY(do_route(c, w, x, W_r, b_r, idx, gates, logits, stream));
  // Forward-only scratch in the backward's buffers.  The T token rows are quantised once (codes and
  // scales in buf_d1, free until the down projection writes o_perm there), and the dispatch gathers
  // their codes and scales into the padded expert rows (in dy_perm: rows x d bytes + 4 rows <=
  // rows x d x 2); the e4m3 h rows and scales go to buf_f1 likewise.
  const size_t rows = (size_t)w.L.rows;
  uint8_t* x8_tok = w.at<uint8_t>(w.L.buf_d1);
  float* xs_tok = reinterpret_cast<float*>(x8_tok + (size_t)c.T * c.d);
  uint8_t* x8 = w.at<uint8_t>(w.L.dy_perm);
  float* xs = reinterpret_cast<float*>(x8 + rows * c.d);
  uint8_t* h8 = w.at<uint8_t>(w.L.buf_f1);
  float* hs = reinterpret_cast<float*>(h8 + rows * c.f);
  uint16_t* h = w.at<uint16_t>(w.L.buf_f0);
  uint16_t* o_perm = w.at<uint16_t>(w.L.buf_d1);
  MOE_CUDA(launch_quantize_rows_e4m3(x, c.T, c.d, x8_tok, xs_tok, stream));
  DispatchArgs da8 = dispatch_args(w);
  da8.idx = idx;
  da8.x = reinterpret_cast<const uint16_t*>(x8_tok);
  da8.x_perm = reinterpret_cast<uint16_t*>(x8);
  da8.xs_tok = xs_tok;
  da8.xs_perm = xs;
  Cfg c8 = c;
  c8.d = c.d / 2;   // an e4m3 row of d codes moves as d / 2 two-byte elements
  MOE_CUDA(launch_dispatch_scan(c, w.L, da8, stream));
  MOE_CUDA(launch_dispatch_gather(c8, w.L, da8, true, true, false, stream));
  GateUpFp8Args ga{x8, xs, wg8, wg_scale, wu8, wu_scale, h, w.hdr(), w.tabs()};
  MOE_CUDA(launch_gate_up_fp8(c, w.L, ga, stream));
  MOE_CUDA(launch_quantize_rows_e4m3(h, (int64_t)rows, c.f, h8, hs, stream, w.tabs()));
  DownFp8Args da{h8, hs, wd8, wd_scale, o_perm, w.hdr(), w.tabs()};
  MOE_CUDA(launch_down_fp8(c, w.L, da, stream));
  CombineArgs ca{o_perm, gates, y, w.tabs(), w.at<int32_t>(w.L.prow_of_slot)};
  MOE_CUDA(launch_combine(c, ca, stream));
  return MOE_OK;
}

moe_status_t moe_layer_fwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                           const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                           moe_bf16* y, void* saved, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x && W_r && W_gate && W_up && W_down && y && saved);
  MOE_NEED(aligned16(x) && aligned16(W_r) && (!b_r || aligned16(b_r)) && aligned16(W_gate) &&
           aligned16(W_up) && aligned16(W_down) && aligned16(y) && aligned16(saved));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  int32_t* idx = static_cast<int32_t*>(saved);
  float* gates = reinterpret_cast<float*>(idx + (size_t)c.T * c.k);
  const SavedLayout sv = saved_layout(c);
  float* logits = sv.logits_bytes ? reinterpret_cast<float*>(static_cast<char*>(saved) + sv.logits_off) : nullptr;
  MOE_TRY(do_route(c, w, x, W_r, b_r, idx, gates, logits, stream));
  // x rows to x_perm, or (gather_in_gemm) the tables only: the gate/up GEMM then gathers the x rows
  // itself from token order (MoEBlaze summary, Methodology item 2: dispatch fused with the FFN)
  uint16_t* x_perm = w.at<uint16_t>(w.L.xperm);
  if (c.gather_in_gemm)
    MOE_TRY(do_dispatch_tables(c, w, idx, nullptr, stream));
  else
    MOE_TRY(do_dispatch(c, w, idx, x, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, x_perm, nullptr,
                        stream));
  uint16_t* o_perm = w.at<uint16_t>(w.L.buf_d1);
  // kept a and b go to `saved`, which lives from this call to the backward; the workspace does not
  uint16_t* a_keep = reinterpret_cast<uint16_t*>(static_cast<char*>(saved) + sv.a_off);
  uint16_t* b_keep = reinterpret_cast<uint16_t*>(static_cast<char*>(saved) + sv.b_off);
  FfnFwdArgs fa{x_perm, W_gate, W_up, W_down, w.at<uint16_t>(w.L.buf_f0), o_perm, w.hdr(), w.tabs(),
                a_keep, b_keep, nullptr, nullptr};
  if (c.gather_in_gemm) {
    fa.x_perm = nullptr;
    fa.x_tok = x;
    fa.tok = w.at<int32_t>(w.L.tok_of_prow);
  }
  MOE_CUDA(launch_ffn_fwd(c, w.L, fa, stream));
  CombineArgs ca{o_perm, gates, y, w.tabs(), w.at<int32_t>(w.L.prow_of_slot)};
  MOE_CUDA(launch_combine(c, ca, stream));
  return MOE_OK;
}

moe_status_t moe_layer_bwd(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                           const moe_bf16* W_gate, const moe_bf16* W_up, const moe_bf16* W_down,
                           const void* saved, const moe_bf16* dy,
                           moe_bf16* dx, float* dW_r, float* db_r,
                           moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                           void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(x && W_r && W_gate && W_up && W_down && saved && dy && dx && dW_r && dW_gate && dW_up && dW_down);
  MOE_NEED(aligned16(x) && aligned16(W_r) && (!b_r || aligned16(b_r)) && aligned16(W_gate) &&
           aligned16(W_up) && aligned16(W_down) && aligned16(saved) && aligned16(dy) && aligned16(dx) &&
           aligned16(dW_r) && (!db_r || aligned16(db_r)) && aligned16(dW_gate) && aligned16(dW_up) &&
           aligned16(dW_down));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  const int32_t* idx = static_cast<const int32_t*>(saved);
  const float* gates = reinterpret_cast<const float*>(idx + (size_t)c.T * c.k);
  // the queues again from the saved idx, the rows' gates, and the x and dy rows -- or (gather_in_gemm)
  // no rows: the GEMMs that read them (dh', the recompute, the weight gradients) gather them
  uint16_t* x_perm = w.at<uint16_t>(w.L.xperm);
  uint16_t* dy_perm = w.at<uint16_t>(w.L.dy_perm);
  if (c.gather_in_gemm)
    MOE_TRY(do_dispatch_tables(c, w, idx, gates, stream));
  else
    MOE_TRY(do_dispatch(c, w, idx, x, dy, gates, nullptr, nullptr, nullptr, nullptr, x_perm, dy_perm, stream));
  uint16_t* dx_perm = w.at<uint16_t>(w.L.buf_d1);
  float* dgates = w.at<float>(w.L.dgates);
  const SavedLayout sv = saved_layout(c);
  const uint16_t* a_kept = reinterpret_cast<const uint16_t*>(static_cast<const char*>(saved) + sv.a_off);
  const uint16_t* b_kept = reinterpret_cast<const uint16_t*>(static_cast<const char*>(saved) + sv.b_off);
  if (c.gather_in_gemm)
    MOE_TRY(do_ffn_bwd(c, w, nullptr, nullptr, W_gate, W_up, W_down, dx_perm, dgates, dW_gate, dW_up, dW_down,
                       a_kept, b_kept, stream, x, dy, w.at<int32_t>(w.L.tok_of_prow)));
  else
    MOE_TRY(do_ffn_bwd(c, w, x_perm, dy_perm, W_gate, W_up, W_down, dx_perm, dgates, dW_gate, dW_up, dW_down,
                       a_kept, b_kept, stream));
  float* dlogits = w.at<float>(w.L.dlogits);
  const float* logits =
      sv.logits_bytes ? reinterpret_cast<const float*>(static_cast<const char*>(saved) + sv.logits_off) : nullptr;
  MOE_TRY(do_router_bwd_saved(c, w, x, logits, idx, gates, dgates, dlogits, dW_r, db_r, stream));
  return do_combine_bwd(c, w, dx_perm, dlogits, W_r, dx, stream, true);
}

moe_status_t moe_quantize_cols_e4m3(const moe_bf16* top, const moe_bf16* bottom, int64_t G, int32_t rows_top,
                                    int32_t rows_bottom, int32_t cols, uint8_t* codes, float* scales,
                                    moe_stream_t stream) {
  MOE_NEED(G >= 0 && G <= 65535 && rows_top >= 1 && rows_bottom >= 0 && cols >= 1);
  const int64_t rows = (int64_t)rows_top + rows_bottom;
  MOE_NEED(rows % 16 == 0 && rows <= 32768 && (int64_t)cols * G <= ((int64_t)1 << 31));
  MOE_NEED((rows_bottom == 0) == (bottom == nullptr));
  MOE_NEED(G == 0 || (top && codes && scales && aligned16(top) && aligned16(codes) && aligned16(scales) &&
                      (!bottom || aligned16(bottom))));
  MOE_TRY(check_device());
  MOE_CUDA(launch_quantize_cols_e4m3(top, bottom, G, rows_top, rows_bottom, cols, codes, scales, stream));
  return MOE_OK;
}

moe_status_t moe_layer_bwd_fp8(const moe_config_t* cfg, const moe_bf16* x, const float* W_r, const float* b_r,
                               const uint8_t* wg8, const float* wg_scale, const uint8_t* wu8, const float* wu_scale,
                               const uint8_t* wdt8, const float* wdt_scale, const uint8_t* wgut8,
                               const float* wgut_scale, const void* saved, const moe_bf16* dy, moe_bf16* dx,
                               float* dW_r, float* db_r, moe_bf16* dW_gate, moe_bf16* dW_up, moe_bf16* dW_down,
                               void* ws, size_t ws_bytes, moe_stream_t stream) {
  Cfg c;
  MOE_TRY(make_cfg(cfg, &c));
  MOE_NEED(cfg->keep_rows == 0);   // every row's a, b are recomputed from the codes
  MOE_NEED(x && W_r && wg8 && wg_scale && wu8 && wu_scale && wdt8 && wdt_scale && wgut8 && wgut_scale && saved &&
           dy && dx && dW_r && dW_gate && dW_up && dW_down);
  MOE_NEED(aligned16(x) && aligned16(W_r) && (!b_r || aligned16(b_r)) && aligned16(wg8) && aligned16(wg_scale) &&
           aligned16(wu8) && aligned16(wu_scale) && aligned16(wdt8) && aligned16(wdt_scale) && aligned16(wgut8) &&
           aligned16(wgut_scale) && aligned16(saved) && aligned16(dy) && aligned16(dx) && aligned16(dW_r) &&
           (!db_r || aligned16(db_r)) && aligned16(dW_gate) && aligned16(dW_up) && aligned16(dW_down));
  Ws w;
  MOE_TRY(get_ws(c, ws, ws_bytes, &w));
  MOE_TRY(check_device());
  const int32_t* idx = static_cast<const int32_t*>(saved);
  const float* gates = reinterpret_cast<const float*>(idx + (size_t)c.T * c.k);
  MOE_TRY(do_dispatch_fp8_bwd(c, w, idx, x, dy, gates, stream));
  float* dgates = w.at<float>(w.L.dgates);
  MOE_TRY(do_ffn_bwd_fp8(c, w, wg8, wg_scale, wu8, wu_scale, wdt8, wdt_scale, wgut8, wgut_scale, dgates, dW_gate,
                         dW_up, dW_down, stream));
  float* dlogits = w.at<float>(w.L.dlogits);
  const SavedLayout sv = saved_layout(c);
  const float* logits =
      sv.logits_bytes ? reinterpret_cast<const float*>(static_cast<const char*>(saved) + sv.logits_off) : nullptr;
  MOE_TRY(do_router_bwd_saved(c, w, x, logits, idx, gates, dgates, dlogits, dW_r, db_r, stream));
  return do_combine_bwd(c, w, w.at<uint16_t>(w.L.buf_d1), dlogits, W_r, dx, stream, true);
}

moe_status_t moe_check_error(void* ws, moe_stream_t stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  Hdr* h = static_cast<Hdr*>(ws);
  int32_t st = 0;
  MOE_CUDA(cudaMemcpy(&st, &h->status, sizeof(st), cudaMemcpyDeviceToHost));
  MOE_CUDA(cudaMemset(&h->status, 0, 2 * sizeof(int32_t)));
  return static_cast<moe_status_t>(st);
}

moe_status_t moe_profile_enable(int32_t on) {
  Profiler& p = profiler();
  std::lock_guard<std::mutex> lock(p.mu);
  p.on = on != 0;
  p.used = 0;
  p.marks.clear();
  for (int i = 0; i < kKCount; ++i) {
    p.total_ms[i] = 0.0;
    p.launches[i] = 0;
  }
  return cuda_status(clock_profile_set(p.on));
}

moe_status_t moe_profile_sm_clock(int32_t kernel, double* mhz) {
  if (kernel < 0 || kernel >= kKCount || mhz == nullptr) return MOE_ERR_INVALID_ARG;
  unsigned long long acc[kKCount][2];
  MOE_CUDA(clock_profile_read(acc));
  *mhz = acc[kernel][1] ? 1000.0 * (double)acc[kernel][0] / (double)acc[kernel][1] : 0.0;
  return MOE_OK;
}

moe_status_t moe_profile_read(int32_t kernel, const char** name, double* total_ms, int32_t* launches) {
  if (kernel < 0 || kernel >= kKCount || name == nullptr || total_ms == nullptr || launches == nullptr)
    return MOE_ERR_INVALID_ARG;
  Profiler& p = profiler();
  std::lock_guard<std::mutex> lock(p.mu);
  if (!p.marks.empty()) {   // fold the recorded pairs into the totals (waits for them)
    for (const auto& m : p.marks) {
      float ms = 0.f;
      if (cudaEventSynchronize(p.pool[m.second.second]) != cudaSuccess ||
          cudaEventElapsedTime(&ms, p.pool[m.second.first], p.pool[m.second.second]) != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      p.total_ms[m.first] += ms;
      p.launches[m.first] += 1;
    }
    p.marks.clear();
    p.used = 0;
  }
  *name = kKernelNames[kernel];
  *total_ms = p.total_ms[kernel];
  *launches = p.launches[kernel];
  return MOE_OK;
}

moe_status_t moe_debug_inject(void* ws, int32_t stall_block, int32_t stall_fill, uint64_t timeout_ns,
                              moe_stream_t stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  Hdr* h = static_cast<Hdr*>(ws);
  const int32_t stall_p1 = stall_block < 0 ? 0 : stall_block + 1;
  const int32_t fill_p1 = stall_fill < 0 ? 0 : stall_fill + 1;
  MOE_CUDA(cudaMemcpyAsync(&h->stall_block_p1, &stall_p1, sizeof(stall_p1), cudaMemcpyHostToDevice, stream));
  MOE_CUDA(cudaMemcpyAsync(&h->stall_fill_p1, &fill_p1, sizeof(fill_p1), cudaMemcpyHostToDevice, stream));
  MOE_CUDA(cudaMemcpyAsync(&h->timeout_ns, &timeout_ns, sizeof(timeout_ns), cudaMemcpyHostToDevice, stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  return MOE_OK;
}

}  // extern "C"
