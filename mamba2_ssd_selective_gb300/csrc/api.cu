// libssd C ABI: argument validation, workspace carving and the launch sequence
// of the forward and backward passes.  Nothing here allocates or synchronises.
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "kernels.h"
#include "ssd.h"

using namespace ssd;

namespace {

// limit of the kernels' bounded hand-off waits, for every later call
std::atomic<unsigned long long> g_wait_limit_ns{sm100::kDefaultWaitLimitNs};

int elem_bytes(int dtype) { return dtype == SSD_BF16 ? 2 : 4; }

ssd_status check_dims(const ssd_dims *d) {
  if (!d) return SSD_ERR_NULL_PTR;
  if (d->batch <= 0 || d->seqlen <= 0 || d->nheads <= 0 || d->headdim <= 0 || d->dstate <= 0 || d->ngroups <= 0 ||
      d->chunk <= 0 || d->n_segments <= 0)
    return SSD_ERR_INVALID_DIMS;
  if (d->d_conv != 4 || d->nheads % d->ngroups != 0) return SSD_ERR_INVALID_DIMS;
  if (d->dtype != SSD_BF16 && d->dtype != SSD_F32) return SSD_ERR_DTYPE;
  if ((long long)d->n_segments * d->chunk > d->seqlen || d->seqlen % ((long long)d->n_segments * d->chunk) != 0)
    return SSD_ERR_SEGMENT_ALIGN;
  if (d->headdim % 8 || d->dstate % 8 || d->headdim > 256 || d->dstate > 256 || d->chunk % 32 || d->chunk > 256 ||
      d->n_segments > 1024)
    return SSD_ERR_UNSUPPORTED;
  // index arithmetic inside kernels uses 32-bit products of (batch, seqlen, heads)
  if ((long long)d->batch * d->seqlen > (1LL << 30) || (long long)d->nheads * d->headdim > (1 << 16) ||
      (long long)d->ngroups * d->dstate > (1 << 16))
    return SSD_ERR_UNSUPPORTED;
  if (d->gated_norm != 0 && d->gated_norm != 1) return SSD_ERR_INVALID_DIMS;
  // the norm kernels hold a group's channels in registers: up to 4096 per group
  if (d->gated_norm && (long long)d->nheads * d->headdim / d->ngroups > 4096) return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

Problem problem_from(const ssd_dims *d) {
  Problem pr{};
  pr.b = d->batch;
  pr.L = d->seqlen;
  pr.H = d->nheads;
  pr.P = d->headdim;
  pr.N = d->dstate;
  pr.G = d->ngroups;
  pr.Q = d->chunk;
  pr.S = d->n_segments;
  pr.Cd = pr.H * pr.P + 2 * pr.G * pr.N;
  pr.nc = pr.L / pr.Q;
  pr.cps = pr.nc / pr.S;
  pr.hpg = pr.H / pr.G;
  pr.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  return pr;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ssd_status check_inputs(const ssd_dims *d, const ssd_inputs *in, Problem &pr) {
  if (!in) return SSD_ERR_NULL_PTR;
  if (!in->x || !in->B || !in->C || !in->dt || !in->dt_bias || !in->A_log || !in->D || !in->conv_w || !in->conv_b)
    return SSD_ERR_NULL_PTR;
  const int eb = elem_bytes(d->dtype);
  const long long vec = 16 / eb;
  const long long HP = (long long)d->nheads * d->headdim, GN = (long long)d->ngroups * d->dstate;
  if (in->x_tok_stride < HP || in->B_tok_stride < GN || in->C_tok_stride < GN || in->dt_tok_stride < d->nheads)
    return SSD_ERR_INVALID_DIMS;
  if (!aligned(in->x, 16) || !aligned(in->B, 16) || !aligned(in->C, 16) || !aligned(in->dt, eb) ||
      in->x_tok_stride % vec || in->B_tok_stride % vec || in->C_tok_stride % vec)
    return SSD_ERR_ALIGNMENT;
  if (!aligned(in->dt_bias, 4) || !aligned(in->A_log, 4) || !aligned(in->D, 4) || !aligned(in->conv_w, 16) ||
      !aligned(in->conv_b, 4) || (in->seq_idx && !aligned(in->seq_idx, 16)) ||
      (in->initial_states && !aligned(in->initial_states, 16)))
    return SSD_ERR_ALIGNMENT;
  // the gated norm: z and its weight exactly when dims ask for it
  if (d->gated_norm) {
    if (!in->z || !in->norm_weight) return SSD_ERR_NULL_PTR;
    if (in->z_tok_stride < HP || !(in->norm_eps >= 0.f) || in->norm_eps > 1e30f) return SSD_ERR_INVALID_DIMS;
    if (!aligned(in->z, 16) || in->z_tok_stride % vec || !aligned(in->norm_weight, 16)) return SSD_ERR_ALIGNMENT;
  } else if (in->z || in->norm_weight) {
    return SSD_ERR_INVALID_DIMS;  // a gate given without dims.gated_norm would be ignored: rejected instead
  }
  pr = problem_from(d);
  pr.x = in->x;
  pr.B = in->B;
  pr.C = in->C;
  pr.dt = in->dt;
  pr.xs = in->x_tok_stride;
  pr.Bs = in->B_tok_stride;
  pr.Cs = in->C_tok_stride;
  pr.dts = in->dt_tok_stride;
  pr.dt_bias = in->dt_bias;
  pr.A_log = in->A_log;
  pr.D = in->D;
  pr.conv_w = in->conv_w;
  pr.conv_b = in->conv_b;
  pr.seq_idx = in->seq_idx;
  pr.init = in->initial_states;
  pr.z = d->gated_norm ? in->z : nullptr;
  pr.zs = in->z_tok_stride;
  pr.norm_w = in->norm_weight;
  pr.norm_eps = in->norm_eps;
  return SSD_OK;
}

Workspace plan_for(const ssd_dims *d, const Problem &pr, bool backward) {
  return plan_workspace(pr, elem_bytes(d->dtype), backward, d->dtype == SSD_BF16 && tc_envelope(pr), d->gated_norm != 0);
}

// ---------------------------------------------------------------- profiling
struct ProfRec {
  const char *name;
  int pair;
};
constexpr int kProfMax = 65536;
bool g_prof_on = false;
cudaEvent_t *g_prof_ev = nullptr;  // 2 * kProfMax events, created on first begin
ProfRec g_prof_rec[kProfMax];
int g_prof_n = 0;

struct ProfScope {
  int idx = -1;
  cudaStream_t s;
  ProfScope(const char *name, cudaStream_t st) : s(st) {
    if (g_prof_on && g_prof_n < kProfMax) {
      idx = g_prof_n++;
      g_prof_rec[idx] = {name, idx};
      cudaEventRecord(g_prof_ev[2 * idx], s);
    }
  }
  ~ProfScope() {
    if (idx >= 0) cudaEventRecord(g_prof_ev[2 * idx + 1], s);
  }
};
#define SSD_LAUNCH(name, call) \
  do {                         \
    ProfScope _ps(name, s);    \
    call;                      \
  } while (0)

ssd_status launch_status() {
  const bool host_err = take_host_error();
  return (cudaPeekAtLastError() == cudaSuccess && !host_err) ? SSD_OK : SSD_ERR_CUDA;
}

template <typename T>
constexpr bool kIsBf16 = std::is_same<T, __nv_bfloat16>::value;

// bf16 activations inside the tensor-core kernels' envelope take the tcgen05
// chunk kernels; everything else (fp32 activations, other shapes) the CUDA-core ones
template <typename T>
bool use_tc(const Problem &pr) {
  return kIsBf16<T> && tc_envelope(pr);
}

// point the problem's decay tables at the workspace
Problem with_tables(const Problem &in, char *ws, const Workspace &w) {
  Problem pr = in;
  float *tab = reinterpret_cast<float *>(ws + w.dtab);
  const size_t n = (size_t)pr.b * pr.H * pr.nc;
  pr.cdec = tab;
  pr.dstart = tab + n;
  pr.dend = tab + 2 * n;
  return pr;
}

// Per-sequence final states of a packed row (ssd_forward_varlen).
struct SeqFinals {
  const int *cu_seqlens = nullptr;
  int nseq = 0;
  float *out = nullptr;
};

template <typename T>
ssd_status forward_impl(const Problem &pr_in, T *y, float *final_state, float *segin_user, char *ws,
                        const Workspace &w, cudaStream_t s, const SeqFinals &sf = SeqFinals()) {
  const Problem pr = with_tables(pr_in, ws, w);
  cudaMemsetAsync(ws + w.status, 0, kStatusBytes, s);  // status word and work counters
  T *u = reinterpret_cast<T *>(ws + w.u);
  float *dtv = reinterpret_cast<float *>(ws + w.dtv), *acs = reinterpret_cast<float *>(ws + w.acs);
  float *cb = reinterpret_cast<float *>(ws + w.cb), *sst = reinterpret_cast<float *>(ws + w.sst);
  float *sext = reinterpret_cast<float *>(ws + w.sext), *ablk = reinterpret_cast<float *>(ws + w.ablk);
  float *segin = segin_user ? segin_user : reinterpret_cast<float *>(ws + w.segin);
  int *status = reinterpret_cast<int *>(ws + w.status);
  const bool tc = use_tc<T>(pr);
  T *const y_out = y;
  // the gated norm: a separate pass over the mixer output (written to the workspace)
  if (pr.z) y = reinterpret_cast<T *>(ws + w.ypre);
  SSD_LAUNCH("conv_fwd", launch_conv_fwd<T>(pr, u, dtv, acs, s));  // and dt_prep
  float *cdec = const_cast<float *>(pr.cdec), *dstart = const_cast<float *>(pr.dstart),
        *dend = const_cast<float *>(pr.dend);
  // the tensor-core chunk-state kernel forms the decay tables in the same launch
  if (!tc) SSD_LAUNCH("decay_tables", launch_decay_tables(pr, acs, cdec, dstart, dend, ablk, s));
  if constexpr (kIsBf16<T>) {
    if (tc)  // CB: inside tc_out
      SSD_LAUNCH("tc_chunk_state", launch_tc_state(pr, u, dtv, acs, sst, cdec, dstart, dend, ablk, status, s));
  }
  if (!tc) {
    SSD_LAUNCH("cb", launch_cb<T>(pr, u, cb, s));
    SSD_LAUNCH("chunk_state", launch_chunk_state<T>(pr, u, dtv, acs, sst, s));
  }
  // the tensor-core path re-forms the local states from Sc in its combine pass
  SSD_LAUNCH("local_pass", launch_local_pass(pr, sst, sext, !tc, s));
  SSD_LAUNCH("seg_scan", launch_seg_scan(pr, sext, ablk, segin, final_state, s));
  if constexpr (kIsBf16<T>) {
    if (tc) {
      __nv_bfloat16 *sin16 = reinterpret_cast<__nv_bfloat16 *>(ws + w.sin16);
      SSD_LAUNCH("combine_state", launch_combine_state(pr, sst, segin, sin16, s));
      SSD_LAUNCH("tc_chunk_out", launch_tc_out(pr, u, dtv, acs, sin16, y, status, s));
    }
  }
  if (!tc) SSD_LAUNCH("chunk_out", launch_chunk_out<T>(pr, u, dtv, acs, cb, sst, segin, y, s));
  if (pr.z) SSD_LAUNCH("gated_norm", launch_gated_norm_fwd<T>(pr, y, y_out, s));
  if (sf.out)  // the chunk states (tensor-core path) or local states (CUDA-core path) are still in sst
    SSD_LAUNCH("seq_finals", launch_seq_finals<T>(pr, u, dtv, acs, sst, !tc, segin, sf.cu_seqlens, sf.nseq, sf.out, s));
  return launch_status();
}

template <typename T>
ssd_status backward_impl(const Problem &pr_in, const T *dy, const float *dfinal, const float *segin_user,
                         const ssd_grads *g, char *ws, const Workspace &w, cudaStream_t s) {
  const Problem pr = with_tables(pr_in, ws, w);
  cudaMemsetAsync(ws + w.status, 0, kStatusBytes, s);  // status word and work counters
  T *u = reinterpret_cast<T *>(ws + w.u);
  float *dtv = reinterpret_cast<float *>(ws + w.dtv), *acs = reinterpret_cast<float *>(ws + w.acs);
  float *cb = reinterpret_cast<float *>(ws + w.cb), *sst = reinterpret_cast<float *>(ws + w.sst);
  float *sext = reinterpret_cast<float *>(ws + w.sext), *ablk = reinterpret_cast<float *>(ws + w.ablk);
  float *dsl = reinterpret_cast<float *>(ws + w.dsl), *gext = reinterpret_cast<float *>(ws + w.gext);
  float *gout = reinterpret_cast<float *>(ws + w.gout), *du = reinterpret_cast<float *>(ws + w.du);
  float *wbuf = reinterpret_cast<float *>(ws + w.w), *tok = reinterpret_cast<float *>(ws + w.tok);
  float *dcp = reinterpret_cast<float *>(ws + w.dcp), *dbp = reinterpret_cast<float *>(ws + w.dbp);
  float *chs = reinterpret_cast<float *>(ws + w.chs), *convp = reinterpret_cast<float *>(ws + w.convp);
  GradOut go{g->dx,           g->dB,           g->dC,           g->ddt,    g->dx_tok_stride,
             g->dB_tok_stride, g->dC_tok_stride, g->ddt_tok_stride, g->dz, g->dz_tok_stride};
  int *status = reinterpret_cast<int *>(ws + w.status);
  const bool tc = use_tc<T>(pr);
  // recompute: conv, dt, CB, chunk states, local segment passes (and the scan)
  SSD_LAUNCH("conv_fwd", launch_conv_fwd<T>(pr, u, dtv, acs, s));  // and dt_prep
  float *cdec = const_cast<float *>(pr.cdec), *dstart = const_cast<float *>(pr.dstart),
        *dend = const_cast<float *>(pr.dend);
  if (!tc) SSD_LAUNCH("decay_tables", launch_decay_tables(pr, acs, cdec, dstart, dend, ablk, s));
  if constexpr (kIsBf16<T>) {
    if (tc)  // CB: in-kernel; the decay tables in the same launch
      SSD_LAUNCH("tc_chunk_state", launch_tc_state(pr, u, dtv, acs, sst, cdec, dstart, dend, ablk, status, s));
  }
  if (!tc) {
    SSD_LAUNCH("cb", launch_cb<T>(pr, u, cb, s));
    SSD_LAUNCH("chunk_state", launch_chunk_state<T>(pr, u, dtv, acs, sst, s));
  }
  // with the forward's segment states given, the tensor-core path needs no local
  // pass (its combine re-forms the local states from Sc)
  if (!tc || !segin_user) SSD_LAUNCH("local_pass", launch_local_pass(pr, sst, sext, !tc, s));
  const float *segin = segin_user;
  if (!segin) {
    float *sg = reinterpret_cast<float *>(ws + w.segin);
    SSD_LAUNCH("seg_scan", launch_seg_scan(pr, sext, ablk, sg, nullptr, s));
    segin = sg;
  }
  // the gated norm's backward: the mixer output is recomputed (it scales with L
  // and is not saved), then dout becomes the mixer output's gradient dy
  if (pr.z) {
    T *ypre = reinterpret_cast<T *>(ws + w.ypre), *dyn = reinterpret_cast<T *>(ws + w.dyn);
    if constexpr (kIsBf16<T>) {
      if (tc) {
        __nv_bfloat16 *sin16 = reinterpret_cast<__nv_bfloat16 *>(ws + w.sin16);
        SSD_LAUNCH("combine_state", launch_combine_state(pr, sst, segin, sin16, s));
        SSD_LAUNCH("tc_chunk_out", launch_tc_out(pr, u, dtv, acs, sin16, ypre, status, s));
      }
    }
    if (!tc) SSD_LAUNCH("chunk_out", launch_chunk_out<T>(pr, u, dtv, acs, cb, sst, segin, ypre, s));
    SSD_LAUNCH("gated_norm_bwd", launch_gated_norm_bwd<T>(pr, ypre, dy, dyn, go, reinterpret_cast<float *>(ws + w.normp),
                                                          g->dnorm_weight, s));
    dy = dyn;
  }
  // reverse boundary scan
  if constexpr (kIsBf16<T>) {
    if (tc) SSD_LAUNCH("tc_chunk_z", launch_tc_z(pr, u, dy, dtv, acs, dsl, status, s));
  }
  if (!tc) SSD_LAUNCH("chunk_z", launch_chunk_z<T>(pr, u, dy, acs, dsl, s));
  // the tensor-core path's backward combine re-forms the local gradients from Z
  // for segments of up to 8 chunks, so the local pass then writes only summaries
  bool write_local = true;
  if constexpr (kIsBf16<T>) {
    if (tc && combine_bwd_local_cps(pr) > 0) write_local = false;
  }
  SSD_LAUNCH("local_rev", launch_local_rev(pr, acs, dsl, gext, write_local, s));
  SSD_LAUNCH("seg_rscan",
             launch_seg_rscan(pr, gext, ablk, dfinal, gout, pr.init ? g->dinitial_states : nullptr, s));
  // chunk gradients
  int vcol_parts = 1, nsub = pr.H, spg = pr.hpg;
  float *sdp = nullptr;  // partial <dS_end, S_in> per chunk and element group, when the combine pass computes it
  if constexpr (kIsBf16<T>) {
    if (tc) {
      __nv_bfloat16 *sin16 = reinterpret_cast<__nv_bfloat16 *>(ws + w.sin16);
      __nv_bfloat16 *dse16 = reinterpret_cast<__nv_bfloat16 *>(ws + w.dse16);
      sdp = reinterpret_cast<float *>(ws + w.sdp);
      SSD_LAUNCH("combine_bwd", launch_combine_bwd(pr, sst, segin, dsl, gout, sin16, dse16, sdp, s));
      SSD_LAUNCH("tc_bwd_row", launch_tc_bwd_row(pr, u, dy, dtv, acs, sin16, dcp, tok, status, s));
      SSD_LAUNCH("tc_bwd_col", launch_tc_bwd_col(pr, u, dy, dtv, acs, dse16, du, dbp, tok, status, s));
      vcol_parts = 1;
      nsub = pr.H / tc_head_subset(pr);
      spg = pr.hpg / tc_head_subset(pr);
    }
  }
  if (!tc) {
    SSD_LAUNCH("chunk_w", launch_chunk_w<T>(pr, u, dy, dtv, acs, cb, wbuf, tok, s));
    SSD_LAUNCH("chunk_dx", launch_chunk_dx<T>(pr, u, dy, dtv, acs, cb, dsl, gout, du, s));
    SSD_LAUNCH("chunk_dcdb",
               launch_chunk_dcdb<T>(pr, u, dy, dtv, acs, wbuf, sst, segin, dsl, gout, dcp, dbp, tok, s));
  }
  SSD_LAUNCH("chunk_dt",
             launch_chunk_dt<T>(pr, u, dy, dtv, acs, sst, segin, dsl, gout, tok, vcol_parts, sdp, scan_groups(pr), go,
                                chs, s));
  // conv backward (it sums the dB / dC partials for the B and C channels) and
  // parameter reductions
  const BcParts bc{dbp, dcp, nsub, spg};
  SSD_LAUNCH("conv_bwd", launch_conv_bwd<T>(pr, du, bc, go, convp, w.ntb, s));
  SSD_LAUNCH("param_reduce", launch_param_reduce(pr, chs, convp, w.ntb, g->ddt_bias, g->dA_log, g->dD, g->dconv_w, g->dconv_b, s));
  return launch_status();
}

// Scratch of ssd_forward_static: a fixed array in the library's device memory,
// so that the call allocates nothing.  Host code must not use the symbol as an
// address; it looks up the device address once per device.
static __device__ __align__(256) unsigned char g_static_scratch[SSD_STATIC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};

// device address of g_static_scratch on the current device (looked up on the
// first call per device), or nullptr on failure
void *static_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
    g_static_ptr[dev] = p;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" {

size_t ssd_workspace_size(const ssd_dims *dims, int backward) {
  if (check_dims(dims) != SSD_OK) return 0;
  const Problem pr = problem_from(dims);
  return plan_for(dims, pr, backward != 0).total;
}

}  // extern "C"

namespace {

// Validation shared by the forward entry points (everything but the scratch).
ssd_status check_forward(const ssd_dims *dims, const ssd_inputs *in, const void *y, const float *final_state,
                         const float *seg_init_states, Problem &pr, Workspace &w) {
  ssd_status st = check_dims(dims);
  if (st != SSD_OK) return st;
  st = check_inputs(dims, in, pr);
  if (st != SSD_OK) return st;
  if (!y) return SSD_ERR_NULL_PTR;
  if (!aligned(y, 16) || (final_state && !aligned(final_state, 16)) ||
      (seg_init_states && !aligned(seg_init_states, 16)))
    return SSD_ERR_ALIGNMENT;
  w = plan_for(dims, pr, false);
  return SSD_OK;
}

ssd_status run_forward(const ssd_dims *dims, const Problem &pr, const Workspace &w, void *y, float *final_state,
                       float *seg_init_states, char *ws, cudaStream_t s, const SeqFinals &sf = SeqFinals()) {
  if (dims->dtype == SSD_BF16)
    return forward_impl<__nv_bfloat16>(pr, static_cast<__nv_bfloat16 *>(y), final_state, seg_init_states, ws, w, s,
                                       sf);
  return forward_impl<float>(pr, static_cast<float *>(y), final_state, seg_init_states, ws, w, s, sf);
}

}  // namespace

extern "C" {

ssd_status ssd_forward(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                       float *seg_init_states, void *workspace, size_t ws_bytes, ssd_stream_t stream) {
  Problem pr;
  Workspace w;
  const ssd_status st = check_forward(dims, in, y, final_state, seg_init_states, pr, w);
  if (st != SSD_OK) return st;
  if (!workspace || ws_bytes < w.total) return SSD_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return SSD_ERR_ALIGNMENT;
  return run_forward(dims, pr, w, y, final_state, seg_init_states, static_cast<char *>(workspace),
                     reinterpret_cast<cudaStream_t>(stream));
}

ssd_status ssd_forward_varlen(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                              float *seg_init_states, const int32_t *cu_seqlens, int32_t nseq,
                              float *seq_final_states, void *workspace, size_t ws_bytes, ssd_stream_t stream) {
  Problem pr;
  Workspace w;
  const ssd_status st = check_forward(dims, in, y, final_state, seg_init_states, pr, w);
  if (st != SSD_OK) return st;
  if (!cu_seqlens || !seq_final_states || !in->seq_idx) return SSD_ERR_NULL_PTR;
  if (nseq <= 0) return SSD_ERR_INVALID_DIMS;
  if (dims->batch != 1) return SSD_ERR_UNSUPPORTED;  // packed rows: one row of sequences
  if (!aligned(cu_seqlens, 4) || !aligned(seq_final_states, 16)) return SSD_ERR_ALIGNMENT;
  if (!workspace || ws_bytes < w.total) return SSD_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return SSD_ERR_ALIGNMENT;
  SeqFinals sf;
  sf.cu_seqlens = cu_seqlens;
  sf.nseq = nseq;
  sf.out = seq_final_states;
  return run_forward(dims, pr, w, y, final_state, seg_init_states, static_cast<char *>(workspace),
                     reinterpret_cast<cudaStream_t>(stream), sf);
}

ssd_status ssd_forward_static(const ssd_dims *dims, const ssd_inputs *in, void *y, float *final_state,
                              float *seg_init_states, ssd_stream_t stream) {
  Problem pr;
  Workspace w;
  const ssd_status st = check_forward(dims, in, y, final_state, seg_init_states, pr, w);
  if (st != SSD_OK) return st;
  if (w.total > SSD_STATIC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
  void *scratch = static_scratch_ptr();
  if (!scratch) return SSD_ERR_CUDA;
  return run_forward(dims, pr, w, y, final_state, seg_init_states, static_cast<char *>(scratch),
                     reinterpret_cast<cudaStream_t>(stream));
}

ssd_status ssd_backward(const ssd_dims *dims, const ssd_inputs *in, const void *dy, const float *dfinal_state,
                        const float *seg_init_states, const ssd_grads *grads, void *workspace, size_t ws_bytes,
                        ssd_stream_t stream) {
  ssd_status st = check_dims(dims);
  if (st != SSD_OK) return st;
  Problem pr;
  st = check_inputs(dims, in, pr);
  if (st != SSD_OK) return st;
  if (!dy || !grads) return SSD_ERR_NULL_PTR;
  if (!grads->dx || !grads->dB || !grads->dC || !grads->ddt || !grads->ddt_bias || !grads->dA_log || !grads->dD ||
      !grads->dconv_w || !grads->dconv_b)
    return SSD_ERR_NULL_PTR;
  if (grads->dinitial_states && !aligned(grads->dinitial_states, 16)) return SSD_ERR_ALIGNMENT;
  const int eb = elem_bytes(dims->dtype);
  const long long vec = 16 / eb;
  const long long HP = (long long)dims->nheads * dims->headdim, GN = (long long)dims->ngroups * dims->dstate;
  if (dims->gated_norm) {
    if (!grads->dz || !grads->dnorm_weight) return SSD_ERR_NULL_PTR;
    if (grads->dz_tok_stride < HP) return SSD_ERR_INVALID_DIMS;
    if (!aligned(grads->dz, 16) || grads->dz_tok_stride % vec || !aligned(grads->dnorm_weight, 4))
      return SSD_ERR_ALIGNMENT;
  }
  if (grads->dx_tok_stride < HP || grads->dB_tok_stride < GN || grads->dC_tok_stride < GN ||
      grads->ddt_tok_stride < dims->nheads)
    return SSD_ERR_INVALID_DIMS;
  if (!aligned(dy, 16) || !aligned(grads->dx, 16) || !aligned(grads->dB, 16) || !aligned(grads->dC, 16) ||
      !aligned(grads->ddt, eb) || grads->dx_tok_stride % vec || grads->dB_tok_stride % vec ||
      grads->dC_tok_stride % vec || (dfinal_state && !aligned(dfinal_state, 16)) ||
      (seg_init_states && !aligned(seg_init_states, 16)))
    return SSD_ERR_ALIGNMENT;
  const Workspace w = plan_for(dims, pr, true);
  if (!workspace || ws_bytes < w.total) return SSD_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return SSD_ERR_ALIGNMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  if (dims->dtype == SSD_BF16)
    return backward_impl<__nv_bfloat16>(pr, static_cast<const __nv_bfloat16 *>(dy), dfinal_state, seg_init_states,
                                        grads, ws, w, s);
  return backward_impl<float>(pr, static_cast<const float *>(dy), dfinal_state, seg_init_states, grads, ws, w, s);
}

ssd_status ssd_cu_seqlens_to_seq_idx(const int32_t *cu_seqlens, int32_t nseq, int32_t *seq_idx,
                                     int32_t total_tokens, ssd_stream_t stream) {
  if (!cu_seqlens || !seq_idx) return SSD_ERR_NULL_PTR;
  if (nseq <= 0 || total_tokens <= 0) return SSD_ERR_INVALID_DIMS;
  if (!aligned(cu_seqlens, 4) || !aligned(seq_idx, 4)) return SSD_ERR_ALIGNMENT;
  launch_cu_seqlens(cu_seqlens, nseq, seq_idx, total_tokens, reinterpret_cast<cudaStream_t>(stream));
  return launch_status();
}

ssd_status ssd_device_status(const void *workspace, ssd_stream_t stream) {
  const void *word = workspace ? workspace : static_scratch_ptr();
  if (!word) return SSD_ERR_CUDA;
  int v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSD_ERR_CUDA;
  return v == 0 ? SSD_OK : SSD_ERR_DEVICE_TIMEOUT;
}

uint64_t ssd_set_wait_limit_ns(uint64_t limit_ns) {
  return g_wait_limit_ns.exchange(limit_ns);
}

ssd_status ssd_profile_begin(void) {
  if (!g_prof_ev) {
    g_prof_ev = new cudaEvent_t[2 * kProfMax];
    for (int i = 0; i < 2 * kProfMax; ++i)
      if (cudaEventCreate(&g_prof_ev[i]) != cudaSuccess) return SSD_ERR_CUDA;
  }
  g_prof_n = 0;
  g_prof_on = true;
  return SSD_OK;
}

int32_t ssd_profile_end(ssd_kernel_time *out, int32_t max_entries) {
  g_prof_on = false;
  if (!g_prof_ev) return 0;
  int n = 0;
  for (int i = 0; i < g_prof_n; ++i) {
    if (cudaEventSynchronize(g_prof_ev[2 * i + 1]) != cudaSuccess) return SSD_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof_ev[2 * i], g_prof_ev[2 * i + 1]) != cudaSuccess) return SSD_ERR_CUDA;
    int j = 0;
    while (j < n && strcmp(out[j].name, g_prof_rec[i].name) != 0) ++j;
    if (j == n) {
      if (n >= max_entries) continue;
      out[n++] = {g_prof_rec[i].name, 0, 0.f};
    }
    out[j].launches += 1;
    out[j].total_ms += ms;
  }
  g_prof_n = 0;
  return n;
}

const char *ssd_status_string(ssd_status status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_DIMS: return "invalid dimensions";
    case SSD_ERR_SEGMENT_ALIGN: return "seqlen is not a multiple of n_segments * chunk";
    case SSD_ERR_NULL_PTR: return "a required pointer is NULL";
    case SSD_ERR_ALIGNMENT: return "pointer or stride misaligned";
    case SSD_ERR_DTYPE: return "unknown activation dtype";
    case SSD_ERR_WORKSPACE: return "workspace missing or too small";
    case SSD_ERR_UNSUPPORTED: return "shape outside the supported envelope";
    case SSD_ERR_CUDA: return "CUDA launch failed";
    case SSD_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
