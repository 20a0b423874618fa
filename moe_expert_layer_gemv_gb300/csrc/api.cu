// api.cu -- the C ABI of include/moe.h: argument validation, workspace
// carve-up, and the launch sequence of each call on the caller's stream.
//
// moe_layer_forward enqueues, all on one stream and chained by programmatic
// dependent launch (no host synchronisation anywhere; the first kernel too may
// start while the stream's previous kernel finishes: it requests only the
// router weights before its griddepcontrol.wait):
//   1. routing: at decode sizes (T <= 128) one launch -- router GEMV over many
//      CTAs, top-k by the last CTA of each token tile; above that, router,
//      top-k and align (+ the workspace plan) as three launches
//   2. gate_up + SwiGLU                  (persistent, bulk-copy pipeline)
//   3. down                              (persistent, bulk-copy pipeline)
//   At decode sizes stages 2 and 3 build the align layout and their work plan
//   from the routing ids in every CTA's shared memory (no serial plan step
//   between the routing and the weight streams); the down stage also leaves
//   the aligned layout in the workspace.
//   4. combine + shared-expert gate      (one CTA per token and column block)
// The shared expert rides in stages 2-3 as one more work expert, so its weight
// stream overlaps the routed experts' ("veloGB10", Kernel work: shared-expert
// work overlapped with the MoE step; small kernels -- the expert routing --
// folded into their neighbours).
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "launch.h"

namespace moe {

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int smem_optin = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.init) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    di.init = true;
  }
  *out = di;
  return true;
}

// Shared-memory budget per CTA of the persistent GEMV kernels: the SM's 228 KB
// split over kCtasPerSm CTAs, less the 1 KB the hardware reserves per CTA and a
// little slack.  Fixed (not read from the device) so that the stage plan, hence
// the unit counts, depend only on the dims.
constexpr int kGemvSmemBudget = 228 * 1024 / kCtasPerSm - 1024 - 512;

struct Layout {
  size_t header, plan, work, cta, logits, sg, htc, ids, w, sorted, blocks, npp, offs, h, hs, y, ys,
      achunk, arank, total;
  int64_t cap;
  bool tc;           // the dims qualify for the tensor-core expert path
  int hs0, h_rows;   // tensor-core path: first shared-expert row of htc, rows of htc
};

// Smallest T routed through the tensor-core grouped GEMMs (below it, the
// weight-streaming GEMVs).
constexpr int kTcMinT = 256;

// Batch-invariant calls stay on the weight-streaming kernels, whose per-token
// arithmetic does not depend on T.
bool invariant(const moe_dims_t& dm) { return (dm.flags & MOE_FLAG_BATCH_INVARIANT) != 0; }

bool tc_dims(const moe_dims_t& dm) {
  return dm.T >= kTcMinT && !invariant(dm) && dm.weight_format == MOE_WEIGHTS_BF16 &&
         dm.block_size % 128 == 0 && dm.I % 128 == 0 && dm.d % 256 == 0 &&
         (dm.I_shared == 0 || dm.I_shared == dm.I);
}

// Router logits on the tensor cores from the same T up.
bool use_tc_router(const moe_dims_t& dm) {
  return dm.T >= kTcMinT && !invariant(dm) && tc_router_supported(dm.T, dm.d, dm.E);
}

size_t carve(size_t* cursor, size_t bytes) {
  const size_t at = *cursor;
  *cursor += (bytes + kAlign - 1) / kAlign * kAlign;
  return at;
}

Layout layout_of(const moe_dims_t& dm) {
  Layout L;
  const int64_t S = (int64_t)dm.T * dm.top_k;
  L.cap = S + (int64_t)dm.E * (dm.block_size - 1);
  size_t c = 0;
  L.header = carve(&c, kAlign);
  L.plan = carve(&c, sizeof(Plan));
  L.work = carve(&c, sizeof(WorkExpert) * (size_t)(dm.E + 1));
  L.cta = carve(&c, sizeof(int32_t) * 4 * ((size_t)kMaxGrid + 1));
  L.logits = carve(&c, sizeof(float) * (size_t)dm.T * dm.E);
  L.sg = carve(&c, sizeof(float) * (size_t)dm.T);
  L.ids = carve(&c, sizeof(int32_t) * (size_t)S);
  L.w = carve(&c, sizeof(float) * (size_t)S);
  L.sorted = carve(&c, sizeof(int32_t) * (size_t)L.cap);
  L.blocks = carve(&c, sizeof(int32_t) * (size_t)(L.cap / dm.block_size + 1));
  L.npp = carve(&c, sizeof(int32_t));
  L.offs = carve(&c, sizeof(int32_t) * (size_t)(dm.E + 1));
  L.achunk = carve(&c, sizeof(int32_t) * (size_t)dm.E * align_chunks(dm.T, dm.top_k));
  L.arank = carve(&c, sizeof(int32_t) * (size_t)S);
  L.h = carve(&c, sizeof(float) * (size_t)L.cap * dm.I);
  L.hs = carve(&c, sizeof(float) * (size_t)dm.T * dm.I_shared);
  L.y = carve(&c, sizeof(float) * (size_t)S * dm.d);
  L.ys = carve(&c, sizeof(float) * (size_t)dm.T * dm.d);
  L.tc = tc_dims(dm);
  L.hs0 = (int)round_up(L.cap, 128);
  L.h_rows = L.hs0 + (int)round_up(dm.T, 128);
  L.htc = carve(&c, L.tc ? sizeof(uint16_t) * (size_t)L.h_rows * dm.I : 0);
  L.total = c;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_dims(const moe_dims_t* dm) {
  if (dm == nullptr) return MOE_ERR_INVALID_ARG;
  const moe_dims_t& d = *dm;
  if (d.T < 0 || d.d <= 0 || d.E <= 0 || d.top_k <= 0 || d.I <= 0 || d.I_shared < 0 ||
      d.block_size <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d.renormalize != 0 && d.renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (d.T > 65536 || d.d < 8 || d.d > 8192 || d.d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (d.E > 1024 || d.top_k > d.E || d.top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (d.I < 8 || d.I > 4096 || d.I % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (d.I_shared != 0 && (d.I_shared < 8 || d.I_shared > 4096 || d.I_shared % 8 != 0))
    return MOE_ERR_UNSUPPORTED;
  if (d.block_size > 1024) return MOE_ERR_UNSUPPORTED;
  if ((d.flags & ~(int32_t)MOE_FLAG_BATCH_INVARIANT) != 0) return MOE_ERR_UNSUPPORTED;
  if (d.weight_format == MOE_WEIGHTS_BF16) return MOE_OK;
  if (d.weight_format == MOE_WEIGHTS_INT4_G32) {
    if (d.group_size != 32 || d.d % 256 != 0 || d.I % 256 != 0) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
  }
  return MOE_ERR_UNSUPPORTED;
}

moe_status_t check_ws(const moe_dims_t& dm, void* ws, size_t ws_bytes, Layout* L) {
  *L = layout_of(dm);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L->total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_weights(const moe_dims_t& dm, const moe_expert_weights_t* ex,
                           const moe_shared_weights_t* sh) {
  if (ex == nullptr || ex->gate_up == nullptr || ex->down == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ex->gate_up) || !aligned16(ex->down)) return MOE_ERR_INVALID_ARG;
  if (dm.weight_format == MOE_WEIGHTS_INT4_G32) {
    if (ex->gate_up_scales == nullptr || ex->down_scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ex->gate_up_scales) || !aligned16(ex->down_scales)) return MOE_ERR_INVALID_ARG;
  }
  if ((sh != nullptr) != (dm.I_shared > 0)) return MOE_ERR_INVALID_ARG;
  if (sh != nullptr) {
    if (sh->gate_up == nullptr || sh->down == nullptr || sh->gate_w == nullptr)
      return MOE_ERR_INVALID_ARG;
    if (!aligned16(sh->gate_up) || !aligned16(sh->down) || !aligned16(sh->gate_w))
      return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

struct ExpertPlan {
  GemvShape gu, dn;
  PlanParams pp;
  bool tc;         // run the expert stages on the tensor cores
  bool smem_plan;  // the GEMV stages plan from the routing ids in shared memory
  int sms;
};

// Routing slots and tokens up to which the GEMV stages may plan in shared
// memory (the token bitmasks of the plan hold up to 128 tokens per expert).
constexpr int kSmemPlanMaxSlots = 2048;
constexpr int kSmemPlanMaxT = 128;

// smem_plan_ok: the caller leaves the routing ids in the workspace and does
// not build a workspace plan, so the GEMV stages may plan for themselves.
moe_status_t expert_plan(const moe_dims_t& dm, void* ws, const Layout& L, int sms,
                         bool smem_plan_ok, ExpertPlan* ep) {
  const int fmt = dm.weight_format;
  const int S = dm.T * dm.top_k;
  ep->smem_plan = false;
  if (smem_plan_ok && !L.tc && S <= kSmemPlanMaxSlots && dm.T <= kSmemPlanMaxT) {
    const int r = smem_plan_bytes(dm.E, S);
    ep->gu = gate_up_shape(fmt, dm.d, dm.I, dm.I_shared, kGemvSmemBudget, r);
    ep->dn = down_shape(fmt, dm.d, dm.I, dm.I_shared, kGemvSmemBudget, r);
    ep->smem_plan = smem_plan_fits(ep->gu, dm.E, dm.T, dm.top_k) &&
                    smem_plan_fits(ep->dn, dm.E, dm.T, dm.top_k);
  }
  if (!ep->smem_plan) {
    ep->gu = gate_up_shape(fmt, dm.d, dm.I, dm.I_shared, kGemvSmemBudget, 0);
    ep->dn = down_shape(fmt, dm.d, dm.I, dm.I_shared, kGemvSmemBudget, 0);
  }
  if (ep->gu.n_stages < 2 || ep->dn.n_stages < 2) return MOE_ERR_UNSUPPORTED;
  PlanParams& pp = ep->pp;
  pp.work = at<WorkExpert>(ws, L.work);
  pp.plan = at<Plan>(ws, L.plan);
  pp.tiles_gu = (int)ceil_div(dm.I, ep->gu.rg);
  pp.tiles_dn = (int)ceil_div(dm.d, ep->dn.rg);
  pp.tiles_gu_shared = dm.I_shared > 0 ? (int)ceil_div(dm.I_shared, ep->gu.rg_shared) : 0;
  pp.tiles_dn_shared = dm.I_shared > 0 ? (int)ceil_div(dm.d, ep->dn.rg_shared) : 0;
  pp.xt_gu = ep->gu.xt;
  pp.xt_dn = ep->dn.xt;
  // Unit costs of the static CTA split, in tokens of arithmetic (chosen by
  // timing the decode layers).  A bf16 gate_up unit streams its weight rows
  // from HBM in about the time of four tokens' arithmetic on them.  A bf16
  // down unit is worth about three: each of its tokens re-reads an h row from
  // shared memory per row pair.  An int4 routed unit runs on the tensor pipe,
  // where up to eight tokens cost what one does: its cost is a constant, about
  // that of a three-token shared-expert gate_up unit (16 + 16 rows against 4
  // row pairs) and of two four-token shared down units (128 rows against 8).
  pp.tok_w = fmt ? 0 : 1;
  // int4 layers number their units tile-major: the re-reads of a weight tile
  // by an expert's further token groups come from L2 (timed: the bf16
  // layers, whose units cost more per token, do better group-major).
  pp.tile_major = fmt ? 1 : 0;
  // Dynamic tails (kStaticShare) pay on long stages only: a stage's end
  // spread is about a tenth of its length, while a tail costs a ticket round
  // trip at the end of every CTA -- and, for gate_up, the down stage's head
  // start (down CTAs plan and start their first weight copies in the SM slots
  // of gate_up CTAs that finish early, about 5 us, lost when every gate_up CTA
  // is kept busy to the end).  So a stage gets a tail when the weight stream
  // of its at most min(E, T k) touched experts reaches 150 MB (down) or 300 MB
  // (gate_up): about 25 and 50 us at the measured HBM rate (timed on the
  // decode layers: verify_t8's down at 134 MB loses with one, int4_t32's at
  // 189 MB gains).
  {
    const double touched = (double)(dm.E < S ? dm.E : S);
    const double gu_bytes =
        touched * (fmt ? 2.0 * dm.I * (dm.d / 2.0 + dm.d / 16.0) : 4.0 * dm.I * dm.d);
    const double dn_bytes =
        touched * (fmt ? (double)dm.d * (dm.I / 2.0 + dm.I / 16.0) : 2.0 * dm.d * dm.I);
    pp.tail_gu = gu_bytes >= 300e6 ? 1 : 0;
    pp.tail_dn = dn_bytes >= 150e6 ? 1 : 0;
  }
  pp.base_gu = fmt ? 7 : 4;
  pp.base_dn = fmt ? 16 : 3;
  pp.base_gu_s = 4;
  pp.base_dn_s = fmt ? 8 : 3;
  ep->sms = sms;
  ep->tc = L.tc && tc_supported(dm.weight_format, dm.d, dm.I, dm.I_shared, dm.block_size);
  pp.tc_nb_gu = ep->tc ? tc_tiles_per_mblock_gu(dm.I) : 0;
  pp.tc_nb_dn = ep->tc ? tc_tiles_per_mblock_dn(dm.d) : 0;
  pp.grid = kCtasPerSm * sms < kMaxGrid ? kCtasPerSm * sms : kMaxGrid;
  pp.cta_gu = at<int32_t>(ws, L.cta);
  pp.cta_dn = at<int32_t>(ws, L.cta) + 2 * (kMaxGrid + 1);
  return MOE_OK;
}

ExpertArgs expert_args(const moe_dims_t& dm, const moe_expert_weights_t* ex,
                       const moe_shared_weights_t* sh) {
  ExpertArgs a;
  a.fmt = dm.weight_format;
  a.gate_up = ex->gate_up;
  a.gate_up_scales = static_cast<const uint16_t*>(ex->gate_up_scales);
  a.down = ex->down;
  a.down_scales = static_cast<const uint16_t*>(ex->down_scales);
  a.s_gate_up = sh ? static_cast<const uint16_t*>(sh->gate_up) : nullptr;
  a.s_down = sh ? static_cast<const uint16_t*>(sh->down) : nullptr;
  a.T = dm.T;
  a.d = dm.d;
  a.E = dm.E;
  a.k = dm.top_k;
  a.I = dm.I;
  a.Is = sh ? dm.I_shared : 0;
  a.h_rows = (int)((int64_t)dm.T * dm.top_k + (int64_t)dm.E * (dm.block_size - 1));
  return a;
}

moe_status_t record(void* const* events, int which, cudaStream_t st) {
  if (events && events[which] &&
      cudaEventRecord(static_cast<cudaEvent_t>(events[which]), st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Stages 3-5 given a plan in the workspace, or (ep.smem_plan) the routing ids
// in the workspace.
moe_status_t run_experts(const moe_dims_t& dm, const void* x, const float* topk_w,
                         const float* sg, const int32_t* sorted_ids, const moe_expert_weights_t* ex,
                         const moe_shared_weights_t* sh, void* out, void* ws, const Layout& L,
                         const ExpertPlan& ep, cudaStream_t st, void* const* events) {
  SmemPlanArgs sp_gu = {}, sp_dn = {};
  if (ep.smem_plan) {
    sp_gu.ids = at<int32_t>(ws, L.ids);
    sp_gu.E = dm.E;
    sp_gu.B = dm.block_size;
    sp_dn = sp_gu;
    sp_gu.base = ep.pp.base_gu;
    sp_gu.base_s = ep.pp.base_gu_s;
    sp_dn.base = ep.pp.base_dn;
    sp_dn.base_s = ep.pp.base_dn_s;
    sp_gu.tok_w = sp_dn.tok_w = ep.pp.tok_w;
    sp_gu.tile_major = sp_dn.tile_major = ep.pp.tile_major;
    sp_gu.tail = ep.pp.tail_gu;
    sp_dn.tail = ep.pp.tail_dn;
    // The down stage leaves the aligned layout in the workspace.
    sp_dn.sorted_ids = at<int32_t>(ws, L.sorted);
    sp_dn.block_ids = at<int32_t>(ws, L.blocks);
    sp_dn.num_post_pad = at<int32_t>(ws, L.npp);
    sp_dn.expert_offsets = at<int32_t>(ws, L.offs);
  }
  const LaunchCfg next{st, true};
  int* status = at<int>(ws, L.header);
  const ExpertArgs a = expert_args(dm, ex, sh);
  float* h = at<float>(ws, L.h);
  float* hs = at<float>(ws, L.hs);
  float* y = at<float>(ws, L.y);
  float* ys = at<float>(ws, L.ys);
  moe_status_t s;
  if (ep.tc) {
    uint16_t* htc = at<uint16_t>(ws, L.htc);
    if (launch_tc(next, false, a, static_cast<const uint16_t*>(x), sorted_ids, ep.pp.plan,
                  ep.pp.work, htc, L.hs0, L.h_rows, y, ys, status, ep.sms) != cudaSuccess)
      return MOE_ERR_CUDA;
    if ((s = record(events, MOE_EV_GATE_UP, st)) != MOE_OK) return s;
    if (launch_tc(next, true, a, static_cast<const uint16_t*>(x), sorted_ids, ep.pp.plan,
                  ep.pp.work, htc, L.hs0, L.h_rows, y, ys, status, ep.sms) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    if (launch_gate_up(next, a, ep.gu, static_cast<const uint16_t*>(x), sorted_ids, ep.pp.plan,
                       ep.pp.work, ep.pp.cta_gu, sp_gu, h, hs, status, ep.pp.grid,
                       ep.pp.tail_gu != 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    if ((s = record(events, MOE_EV_GATE_UP, st)) != MOE_OK) return s;
    if (launch_down(next, a, ep.dn, sorted_ids, ep.pp.plan, ep.pp.work, ep.pp.cta_dn, sp_dn, h, hs,
                    y, ys, status, ep.pp.grid, ep.pp.tail_dn != 0) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if ((s = record(events, MOE_EV_DOWN, st)) != MOE_OK) return s;
  if (launch_combine(next, dm.T, dm.d, dm.top_k, topk_w, y, sh ? ys : nullptr, sh ? sg : nullptr,
                     static_cast<const uint16_t*>(x),
                     sh ? static_cast<const uint16_t*>(sh->gate_w) : nullptr,
                     static_cast<uint16_t*>(out)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace

moe_status_t layer_precheck(const moe_dims_t* dims, const void* x, const void* router_w,
                            const moe_expert_weights_t* ex, const moe_shared_weights_t* sh,
                            const void* out, const void* ids_out, const void* w_out) {
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK || dims->T == 0) return s;
  if (x == nullptr || router_w == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if ((ids_out && !aligned16(ids_out)) || (w_out && !aligned16(w_out))) return MOE_ERR_INVALID_ARG;
  return check_weights(*dims, ex, sh);
}

namespace {

moe_status_t layer_forward(const moe_dims_t* dims, const void* x, const void* router_w,
                           const moe_expert_weights_t* ex, const moe_shared_weights_t* sh,
                           void* out, int32_t* ids_out, float* w_out, void* ws, size_t ws_bytes,
                           void* stream, void* const* events) {
  moe_status_t s = layer_precheck(dims, x, router_w, ex, sh, out, ids_out, w_out);
  if (s != MOE_OK) return s;
  const moe_dims_t dm = *dims;
  if (dm.T == 0) return MOE_OK;  // no tokens: nothing read, written or launched
  Layout L;
  if ((s = check_ws(dm, ws, ws_bytes, &L)) != MOE_OK) return s;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  const bool fused = fused_route_supported(dm.T, dm.E, dm.top_k);
  ExpertPlan ep;
  if ((s = expert_plan(dm, ws, L, di.sms, fused, &ep)) != MOE_OK) return s;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LaunchCfg next{st, true};
  int* status = at<int>(ws, L.header);
  float* logits = at<float>(ws, L.logits);
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* w = at<float>(ws, L.w);
  int32_t* sorted = at<int32_t>(ws, L.sorted);

  if ((s = record(events, MOE_EV_BEGIN, st)) != MOE_OK) return s;
  const uint16_t* w_sg = sh ? static_cast<const uint16_t*>(sh->gate_w) : nullptr;
  float* sg = at<float>(ws, L.sg);
  if (fused) {
    if (launch_route_fused(next, static_cast<const uint16_t*>(x),
                           static_cast<const uint16_t*>(router_w), w_sg, logits, sg, dm.T, dm.d,
                           dm.E, dm.top_k, dm.renormalize, ids, w, ids_out, w_out, !ep.smem_plan,
                           dm.block_size, sorted, at<int32_t>(ws, L.blocks), at<int32_t>(ws, L.npp),
                           at<int32_t>(ws, L.offs), ep.pp, status, status + kRouteCounterBase,
                           di.sms) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    // After the tensor-core router the top-k kernel also takes the
    // shared-expert gate logit x . w_sg (one warp per token).
    const bool tc_router = use_tc_router(dm);
    if (tc_router) {
      if (launch_tc_router(next, static_cast<const uint16_t*>(x),
                           static_cast<const uint16_t*>(router_w), logits, dm.T, dm.d, dm.E,
                           status, di.sms) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else if (launch_router_logits(next, static_cast<const uint16_t*>(x),
                                    static_cast<const uint16_t*>(router_w), w_sg, logits, sg,
                                    dm.T, dm.d, dm.E, di.sms, status) != cudaSuccess) {
      return MOE_ERR_CUDA;
    }
    if (launch_topk(next, logits, dm.T, dm.E, dm.top_k, dm.renormalize, ids, w, ids_out, w_out,
                    static_cast<const uint16_t*>(x), dm.d, tc_router ? w_sg : nullptr,
                    tc_router ? sg : nullptr) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (launch_align(next, ids, dm.T, dm.E, dm.top_k, dm.block_size, sorted,
                     at<int32_t>(ws, L.blocks), at<int32_t>(ws, L.npp), at<int32_t>(ws, L.offs),
                     ep.pp, status, at<int32_t>(ws, L.achunk), at<int32_t>(ws, L.arank),
                     status + kAlignCounter) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if ((s = record(events, MOE_EV_ROUTED, st)) != MOE_OK) return s;
  if ((s = run_experts(dm, x, w, sg, sorted, ex, sh, out, ws, L, ep, st, events)) != MOE_OK)
    return s;
  return record(events, MOE_EV_END, st);
}

}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {
__global__ void set_word_kernel(int* word, int value) { *word = value; }
}  // namespace

cudaError_t launch_set_word(const LaunchCfg& c, int* word, int value) {
  void* args[] = {&word, &value};
  return launch_kernel(c, (const void*)set_word_kernel, dim3(1), dim3(1), 0, args);
}

cudaError_t launch_kernel(const LaunchCfg& c, const void* fn, dim3 grid, dim3 block, size_t smem,
                          void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = c.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t ensure_smem(const void* fn, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::unordered_map<const void*, int> set_to[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = set_to[dev].find(fn);
  if (it != set_to[dev].end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) set_to[dev][fn] = bytes;
  return e;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer, misalignment or bad value";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: dims outside the supported limits";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK: a kernel saw an out-of-range index";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a kernel's bounded pipeline wait ran out";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_bytes(const moe_dims_t* dims, size_t* bytes) {
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = 0;
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK) return s;
  *bytes = layout_of(*dims).total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < kAlign)
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, kAlign, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_workspace_views(const moe_dims_t* dims, moe_workspace_views_t* views) {
  if (views == nullptr) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK) return s;
  const Layout L = layout_of(*dims);
  views->topk_ids = L.ids;
  views->topk_weights = L.w;
  views->sorted_ids = L.sorted;
  views->block_expert_ids = L.blocks;
  views->num_post_pad = L.npp;
  views->expert_offsets = L.offs;
  return MOE_OK;
}

moe_status_t moe_workspace_inject_stall(void* workspace, size_t workspace_bytes,
                                        uint32_t wait_limit_us, void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0 ||
      workspace_bytes < kAlign)
    return MOE_ERR_WORKSPACE;
  if (wait_limit_us < 1 || wait_limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_set_word(LaunchCfg{static_cast<cudaStream_t>(stream), false},
                                     static_cast<int*>(workspace) + kStallWord,
                                     (int)wait_limit_us));
}

moe_status_t moe_route(const moe_dims_t* dims, const void* x, const void* router_w,
                       int32_t* topk_ids, float* topk_weights, void* workspace,
                       size_t workspace_bytes, void* stream) {
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK) return s;
  const moe_dims_t dm = *dims;
  if (dm.T == 0) return MOE_OK;
  if (!x || !router_w || !topk_ids || !topk_weights) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(topk_ids) || !aligned16(topk_weights))
    return MOE_ERR_INVALID_ARG;
  Layout L;
  if ((s = check_ws(dm, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  if (dm.T == 0) return MOE_OK;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* logits = at<float>(workspace, L.logits);
  const cudaError_t err =
      use_tc_router(dm)
          ? launch_tc_router(LaunchCfg{st, true}, static_cast<const uint16_t*>(x),
                             static_cast<const uint16_t*>(router_w), logits, dm.T, dm.d, dm.E,
                             at<int>(workspace, L.header), di.sms)
          : launch_router_logits(LaunchCfg{st, true}, static_cast<const uint16_t*>(x),
                                 static_cast<const uint16_t*>(router_w), nullptr, logits, nullptr,
                                 dm.T, dm.d, dm.E, di.sms, at<int>(workspace, L.header));
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_topk(LaunchCfg{st, true}, logits, dm.T, dm.E, dm.top_k,
                                 dm.renormalize, topk_ids, topk_weights, nullptr, nullptr,
                                 nullptr, dm.d, nullptr, nullptr));
}

moe_status_t moe_align_block_size(const moe_dims_t* dims, const int32_t* topk_ids,
                                  int32_t* sorted_ids, int32_t* block_expert_ids,
                                  int32_t* num_post_pad, int32_t* expert_offsets, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK) return s;
  const moe_dims_t dm = *dims;
  if (!topk_ids && dm.T > 0) return MOE_ERR_INVALID_ARG;
  if (!sorted_ids || !block_expert_ids || !num_post_pad || !expert_offsets)
    return MOE_ERR_INVALID_ARG;
  if ((topk_ids && !aligned16(topk_ids)) || !aligned16(sorted_ids) || !aligned16(block_expert_ids) ||
      !aligned16(num_post_pad) || !aligned16(expert_offsets))
    return MOE_ERR_INVALID_ARG;
  Layout L;
  if ((s = check_ws(dm, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  PlanParams none = {};
  return cuda_status(launch_align(LaunchCfg{static_cast<cudaStream_t>(stream), true}, topk_ids,
                                  dm.T, dm.E, dm.top_k, dm.block_size, sorted_ids,
                                  block_expert_ids, num_post_pad, expert_offsets, none,
                                  at<int>(workspace, L.header), at<int32_t>(workspace, L.achunk),
                                  at<int32_t>(workspace, L.arank),
                                  at<int>(workspace, L.header) + kAlignCounter));
}

moe_status_t moe_expert_forward(const moe_dims_t* dims, const void* x, const float* topk_weights,
                                const int32_t* sorted_ids, const int32_t* block_expert_ids,
                                const int32_t* num_post_pad, const int32_t* expert_offsets,
                                const moe_expert_weights_t* experts,
                                const moe_shared_weights_t* shared, void* out, void* workspace,
                                size_t workspace_bytes, void* stream) {
  moe_status_t s = check_dims(dims);
  if (s != MOE_OK) return s;
  const moe_dims_t dm = *dims;
  if (dm.T == 0) return MOE_OK;
  if (!x || !topk_weights || !sorted_ids || !block_expert_ids || !num_post_pad ||
      !expert_offsets || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_weights) || !aligned16(sorted_ids) ||
      !aligned16(num_post_pad) || !aligned16(expert_offsets) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if ((s = check_weights(dm, experts, shared)) != MOE_OK) return s;
  Layout L;
  if ((s = check_ws(dm, workspace, workspace_bytes, &L)) != MOE_OK) return s;
  DeviceInfo di;
  if (!device_info(&di)) return MOE_ERR_CUDA;
  ExpertPlan ep;
  if ((s = expert_plan(dm, workspace, L, di.sms, false, &ep)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_plan(LaunchCfg{st, true}, dm.T, dm.E, dm.top_k, dm.block_size, sorted_ids,
                  num_post_pad, expert_offsets, ep.pp, at<int>(workspace, L.header)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return run_experts(dm, x, topk_weights, nullptr, sorted_ids, experts, shared, out, workspace, L,
                     ep, st, nullptr);
}

moe_status_t moe_layer_forward(const moe_dims_t* dims, const void* x, const void* router_w,
                               const moe_expert_weights_t* experts,
                               const moe_shared_weights_t* shared, void* out,
                               int32_t* topk_ids_out, float* topk_weights_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return layer_forward(dims, x, router_w, experts, shared, out, topk_ids_out, topk_weights_out,
                       workspace, workspace_bytes, stream, nullptr);
}

moe_status_t moe_layer_forward_timed(const moe_dims_t* dims, const void* x, const void* router_w,
                                     const moe_expert_weights_t* experts,
                                     const moe_shared_weights_t* shared, void* out,
                                     int32_t* topk_ids_out, float* topk_weights_out,
                                     void* workspace, size_t workspace_bytes, void* stream,
                                     void* const* events) {
  if (events == nullptr) return MOE_ERR_INVALID_ARG;
  return layer_forward(dims, x, router_w, experts, shared, out, topk_ids_out, topk_weights_out,
                       workspace, workspace_bytes, stream, events);
}

moe_status_t moe_read_device_status(void* workspace, int32_t* code, void* stream) {
  if (workspace == nullptr || code == nullptr ||
      (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  if (v != 0 && cudaMemsetAsync(workspace, 0, sizeof v, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
