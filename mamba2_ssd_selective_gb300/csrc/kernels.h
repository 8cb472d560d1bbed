// Host-side launchers of the libssd kernels (internal; not part of the ABI).
#pragma once

#include "common.cuh"
#include "tc_pipe.cuh"

namespace ssd {

struct GradOut {  // raw-input gradient destinations (activation dtype)
  void *dx, *dB, *dC, *ddt;
  long long dxs, dBs, dCs, ddts;
  void *dz;  // the gate's gradient (gated RMSNorm), token stride dzs
  long long dzs;
};

// conv + dt (conv_dt.cu)
// conv + SiLU forward, with the dt preparation (dt and the chunk-local Acs) in the same launch
template <typename T> void launch_conv_fwd(const Problem &pr, T *u, float *dtv, float *acs, cudaStream_t s);
// dB / dC of the post-conv B and C channels as fixed-order sums of per-head-block
// partials (b, L, nsub, N): the partials of group g are [g * spg, (g + 1) * spg)
struct BcParts {
  const float *dbp, *dcp;
  int nsub, spg;
};
// du: the x channels' gradient (b, L, Cd; the B/C columns are not read)
template <typename T>
void launch_conv_bwd(const Problem &pr, const float *du, const BcParts &bc, const GradOut &go, float *convp, int ntb,
                     cudaStream_t s);
void launch_param_reduce(const Problem &pr, const float *chs, const float *convp, int ntb, float *ddt_bias,
                         float *dA_log, float *dD, float *dconv_w, float *dconv_b, cudaStream_t s);
void launch_cu_seqlens(const int *cu, int nseq, int *seq_idx, int total, cudaStream_t s);

// gated RMSNorm after the mixer (norm.cu): out = norm(ypre * silu(z)) * w, and its
// backward (dy, dz, and the norm weight's gradient via per-tile partials dwp)
template <typename T> void launch_gated_norm_fwd(const Problem &pr, const T *ypre, T *y, cudaStream_t s);
template <typename T>
void launch_gated_norm_bwd(const Problem &pr, const T *ypre, const T *dout, T *dy, const GradOut &go, float *dwp,
                           float *dnorm_w, cudaStream_t s);

// segment summaries and scans (scan.cu)
void launch_decay_tables(const Problem &pr, const float *acs, float *cdec, float *dstart, float *dend, float *ablk,
                         cudaStream_t s);
// sc: the chunk states Sc (the local states are re-formed inside)
void launch_combine_state(const Problem &pr, const float *sc, const float *segin, __nv_bfloat16 *out, cudaStream_t s);
void launch_combine_bwd(const Problem &pr, const float *sc, const float *segin, const float *dsl, const float *gout,
                        __nv_bfloat16 *sin16, __nv_bfloat16 *dse16, float *sdp, cudaStream_t s);
void launch_local_pass(const Problem &pr, float *sst, float *sext, bool write_local, cudaStream_t s);
void launch_seg_scan(const Problem &pr, const float *sext, const float *ablk, float *segin, float *final_state,
                     cudaStream_t s);
// write_local: overwrite dsl's Z with the local gradients at the chunk ends
// (else only the segment summaries gext are written)
void launch_local_rev(const Problem &pr, const float *acs, float *dsl, float *gext, bool write_local,
                      cudaStream_t s);
// chunks per segment up to which the backward combine re-forms the local
// gradients from Z itself (0: it reads them as the local pass wrote them)
int combine_bwd_local_cps(const Problem &pr);
void launch_seg_rscan(const Problem &pr, const float *gext, const float *ablk, const float *dfinal, float *gout,
                      float *dinit, cudaStream_t s);
// per-sequence final states of a packed row (varlen.cu); sst_local: sst holds
// the local states entering each chunk (CUDA-core path) rather than the chunk
// states Sc (tensor-core path)
template <typename T>
void launch_seq_finals(const Problem &pr, const T *u, const float *dtv, const float *acs, const float *sst,
                       bool sst_local, const float *segin, const int *cu_seqlens, int nseq, float *out,
                       cudaStream_t s);

// fp32 SIMT chunk kernels (simt_chunk.cu)
template <typename T> void launch_cb(const Problem &pr, const T *u, float *cb, cudaStream_t s);
template <typename T>
void launch_chunk_state(const Problem &pr, const T *u, const float *dtv, const float *acs, float *sst, cudaStream_t s);
template <typename T>
void launch_chunk_out(const Problem &pr, const T *u, const float *dtv, const float *acs, const float *cb,
                      const float *sst, const float *segin, T *y, cudaStream_t s);
template <typename T>
void launch_chunk_z(const Problem &pr, const T *u, const T *dy, const float *acs, float *dsl, cudaStream_t s);
template <typename T>
void launch_chunk_w(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs, const float *cb,
                    float *wbuf, float *tok, cudaStream_t s);
template <typename T>
void launch_chunk_dx(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs, const float *cb,
                     const float *dsl, const float *gout, float *du, cudaStream_t s);
template <typename T>
void launch_chunk_dcdb(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs,
                       const float *wbuf, const float *sst, const float *segin, const float *dsl, const float *gout,
                       float *dcp, float *dbp, float *tok, cudaStream_t s);
template <typename T>
void launch_chunk_dt(const Problem &pr, const T *u, const T *dy, const float *dtv, const float *acs,
                     const float *sst, const float *segin, const float *dsl, const float *gout, const float *tok,
                     int vcol_parts, const float *sdp, int sdp_groups, const GradOut &go, float *chs,
                     cudaStream_t s);

// bf16 tensor-core chunk kernels (tc_chunk.cu); envelope: see tc_envelope()
inline bool tc_envelope(const Problem &pr) {
  return pr.P == 64 && pr.N == 128 && (pr.Q == 128 || pr.Q == 256) && pr.hpg % 2 == 0;
}
// the chunk states, and the decay tables (as launch_decay_tables) in the same launch
void launch_tc_state(const Problem &pr, const __nv_bfloat16 *u, const float *dtv, const float *acs, float *sst,
                     float *cdec, float *dstart, float *dend, float *ablk, int *status, cudaStream_t s);
// persistent output kernel (tc_out.cu): the mixer output y (the gated norm, when
// asked for, is a separate pass over it)
void launch_tc_out(const Problem &pr, const __nv_bfloat16 *u, const float *dtv, const float *acs,
                   const __nv_bfloat16 *sin16, __nv_bfloat16 *y, int *status, cudaStream_t s);
void launch_tc_z(const Problem &pr, const __nv_bfloat16 *u, const __nv_bfloat16 *dy, const float *dtv,
                 const float *acs, float *dsl, int *status, cudaStream_t s);
// persistent backward kernels (tc_bwd_row.cu, tc_bwd_col.cu)
void launch_tc_bwd_row(const Problem &pr, const __nv_bfloat16 *u, const __nv_bfloat16 *dy, const float *dtv,
                       const float *acs, const __nv_bfloat16 *sin16, float *dcp, float *tok, int *status,
                       cudaStream_t s);
void launch_tc_bwd_col(const Problem &pr, const __nv_bfloat16 *u, const __nv_bfloat16 *dy, const float *dtv,
                       const float *acs, const __nv_bfloat16 *dse16, float *du, float *dbp, float *tok, int *status,
                       cudaStream_t s);
int tc_head_subset(const Problem &pr);  // heads per dB/dC partial on the tensor-core path

}  // namespace ssd
