/*
 * ssd_oracle.c -- fp64 CPU oracle for the Mamba2 SSD mixer core.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this library.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes, for one batch row, token by token (no chunking, no
 * blocking, no reordering):
 *
 *   conv + SiLU  (Mamba2 "xBC" depthwise causal conv, width 4; the conv has to
 *                be handled at segment boundaries: state-spaces/mamba issue
 *                #482 "Sequence parallelism in the mixer", comment 2; the halo
 *                is the previous segment's last tokens: Megatron-LM PR #6808
 *                "Add state-passing context parallelism for Mamba2",
 *                description)
 *       v[t,c] = conv_b[c] + sum_{k=0..3} w[c,k] * xr[t-3+k, c]
 *                (taps before token 0 or in another packed sequence are zero)
 *       u[t,c] = v * sigmoid(v)
 *   dt / decay
 *       dt_t = softplus(dt_raw[t,h] + dt_bias[h]),  A = -exp(A_log[h])
 *       a_t  = 0 if the state is reset before token t, else exp(dt_t * A)
 *   state-space recurrence (Mamba2 selective SSM), per head h, group g(h)
 *       h_t = a_t * h_{t-1} + dt_t * x_t (outer) B_t            (P x N)
 *       y_t = h_t . C_t + D[h] * x_t
 *   causal segments (Megatron-LM PR #6808, description: the SSD over one
 *   causal segment is affine in its initial state, S_out = a_block*S_in +
 *   S_ext; each segment computes (S_ext, a_block) from a zero initial state,
 *   an exclusive causal scan over the summaries recovers the true initial
 *   state, and a correction applies it)
 *       S_ext[k]  = state at the end of segment k run from zero
 *       a_block[k]= product of a_t over the segment's tokens
 *       S_in[0]   = 0,  S_in[k] = a_block[k-1]*S_in[k-1] + S_ext[k-1]
 *       y_t      += (prod_{tau=seg start..t} a_tau) * C_t . S_in[k]
 *   resets at packed-sequence boundaries (seq_idx from cu_seqlens:
 *   NeMo Automodel PR #1441 "feat: context-parallel with nemotron v3",
 *   Key changes): reset(t) = (t == 0) or seq_idx[t] != seq_idx[t-1].
 *   Initial states (listed as not supported yet in the Megatron-LM PR's
 *   description; read here as in the Mamba2 chunked scan): the state before a
 *   row's first token is init[h] instead of zero, so token 0 is then no reset
 *   and its decay applies to init; later packed sequences still start from
 *   zero.  In the segmented variant the exclusive scan starts from it:
 *   S_in[0] = init.  The state after the last token of every packed sequence
 *   is available as well (orc_seq_finals).
 *
 *   Backward: the adjoint of the recurrence run in reverse (the reverse
 *   boundary scan of the Megatron-LM PR), with states recomputed from
 *   checkpoints every 256 tokens; then SiLU and conv backward.
 *
 * Everything is fp64.  Work is split over heads (and channels) with pthreads;
 * each task writes disjoint memory and cross-head sums are taken in fixed head
 * order afterwards, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define DCONV 4
#define CKPT 256

typedef struct {
  int L, H, P, N, G;
  const double *xBC;     /* L x Cd raw conv input, channels [x (H*P) | B (G*N) | C (G*N)] */
  const double *dt_raw;  /* L x H */
  const double *dt_bias; /* H */
  const double *A_log;   /* H */
  const double *D;       /* H */
  const double *conv_w;  /* Cd x 4, tap 3 multiplies the current token */
  const double *conv_b;  /* Cd */
  const int *seq_idx;    /* L, non-decreasing, or NULL */
  const double *init;    /* H x P x N: the state before token 0, or NULL (zero) */
} orc_row;

/* ------------------------------------------------------------------ */
/* small helpers                                                       */

static int conv_dim(const orc_row *r) { return r->H * r->P + 2 * r->G * r->N; }

static double softplus(double z) { return z > 0 ? z + log1p(exp(-z)) : log1p(exp(z)); }

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

static int is_reset(const orc_row *r, int t) {
  if (t == 0) return r->init == NULL;
  return r->seq_idx != NULL && r->seq_idx[t] != r->seq_idx[t - 1];
}

static int same_seq(const orc_row *r, int s, int t) {
  return r->seq_idx == NULL || r->seq_idx[s] == r->seq_idx[t];
}

static double dt_of(const orc_row *r, int t, int h) {
  return softplus(r->dt_raw[(size_t)t * r->H + h] + r->dt_bias[h]);
}

static double decay_of(const orc_row *r, int t, int h, double dt) {
  double A = -exp(r->A_log[h]);
  return is_reset(r, t) ? 0.0 : exp(dt * A);
}

/* ------------------------------------------------------------------ */
/* a tiny task pool: tasks write disjoint memory, so order is irrelevant */

typedef struct {
  void (*fn)(void *, int);
  void *ctx;
  int ntasks;
  int next;
  pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg) {
  pool_t *pl = (pool_t *)arg;
  for (;;) {
    pthread_mutex_lock(&pl->mu);
    int i = pl->next++;
    pthread_mutex_unlock(&pl->mu);
    if (i >= pl->ntasks) break;
    pl->fn(pl->ctx, i);
  }
  return NULL;
}

int orc_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void run_tasks(void (*fn)(void *, int), void *ctx, int ntasks, int nthreads) {
  if (nthreads <= 0) nthreads = orc_default_threads();
  if (nthreads > ntasks) nthreads = ntasks;
  if (nthreads <= 1) {
    for (int i = 0; i < ntasks; ++i) fn(ctx, i);
    return;
  }
  pool_t pl;
  pl.fn = fn;
  pl.ctx = ctx;
  pl.ntasks = ntasks;
  pl.next = 0;
  pthread_mutex_init(&pl.mu, NULL);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, pool_worker, &pl);
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
  free(th);
  pthread_mutex_destroy(&pl.mu);
}

/* ------------------------------------------------------------------ */
/* channel subsets: the x channels of heads [h0,h1) followed by the B and  */
/* C channels of the groups those heads use, [g0,g1).                       */

typedef struct {
  int h0, h1, g0, g1;
  int nx, ng, nsub;
} chan_set;

static chan_set make_set(const orc_row *r, int h0, int h1) {
  chan_set s;
  int hpg = r->H / r->G;
  s.h0 = h0;
  s.h1 = h1;
  s.g0 = h0 / hpg;
  s.g1 = (h1 - 1) / hpg + 1;
  s.nx = (h1 - h0) * r->P;
  s.ng = s.g1 - s.g0;
  s.nsub = s.nx + 2 * s.ng * r->N;
  return s;
}

/* global channel index of subset channel j */
static int set_channel(const orc_row *r, const chan_set *s, int j) {
  int GN = r->G * r->N, HP = r->H * r->P;
  if (j < s->nx) return s->h0 * r->P + j;
  j -= s->nx;
  int ngN = s->ng * r->N;
  if (j < ngN) return HP + s->g0 * r->N + j;
  j -= ngN;
  return HP + GN + s->g0 * r->N + j;
}

/* conv + SiLU of one channel: v (pre-activation) and u, both L long */
static void conv_channel(const orc_row *r, int c, double *v, double *u) {
  int Cd = conv_dim(r);
  for (int t = 0; t < r->L; ++t) {
    double acc = r->conv_b[c];
    for (int k = 0; k < DCONV; ++k) {
      int s = t - (DCONV - 1) + k;
      if (s < 0 || !same_seq(r, s, t)) continue;
      acc += r->conv_w[(size_t)c * DCONV + k] * r->xBC[(size_t)s * Cd + c];
    }
    if (v) v[t] = acc;
    u[t] = acc * sigmoid(acc);
  }
}

typedef struct {
  const orc_row *r;
  const chan_set *s;
  double *v; /* nsub x L (channel-major) or NULL */
  double *u; /* nsub x L */
} conv_ctx;

static void conv_task(void *vc, int j) {
  conv_ctx *c = (conv_ctx *)vc;
  size_t L = (size_t)c->r->L;
  conv_channel(c->r, set_channel(c->r, c->s, j), c->v ? c->v + j * L : NULL, c->u + j * L);
}

/* Public: conv + SiLU for the channel subset of heads [h0,h1).
 * u, v: nsub x L, channel-major (v may be NULL).  Returns nsub. */
int orc_conv(const orc_row *r, int h0, int h1, double *u, double *v, int nthreads) {
  chan_set s = make_set(r, h0, h1);
  conv_ctx c = {r, &s, v, u};
  run_tasks(conv_task, &c, s.nsub, nthreads);
  return s.nsub;
}

int orc_subset_size(const orc_row *r, int h0, int h1) { return make_set(r, h0, h1).nsub; }

int orc_subset_channel(const orc_row *r, int h0, int h1, int j) {
  chan_set s = make_set(r, h0, h1);
  return set_channel(r, &s, j);
}

/* pointers into a channel-major subset array for head h / group g */
static const double *sub_x(const orc_row *r, const chan_set *s, const double *base, int h, int p) {
  return base + ((size_t)(h - s->h0) * r->P + p) * r->L;
}
static const double *sub_B(const orc_row *r, const chan_set *s, const double *base, int g, int n) {
  return base + ((size_t)s->nx + (size_t)(g - s->g0) * r->N + n) * r->L;
}
static const double *sub_C(const orc_row *r, const chan_set *s, const double *base, int g, int n) {
  return base + ((size_t)s->nx + (size_t)s->ng * r->N + (size_t)(g - s->g0) * r->N + n) * r->L;
}

/* gather token-major copies (L x P, L x N, L x N) of one head's operands */
static void gather_head(const orc_row *r, const chan_set *s, const double *u, int h, double *x,
                        double *B, double *C) {
  int L = r->L, P = r->P, N = r->N, g = h / (r->H / r->G);
  for (int p = 0; p < P; ++p) {
    const double *src = sub_x(r, s, u, h, p);
    for (int t = 0; t < L; ++t) x[(size_t)t * P + p] = src[t];
  }
  for (int n = 0; n < N; ++n) {
    const double *sb = sub_B(r, s, u, g, n), *sc = sub_C(r, s, u, g, n);
    for (int t = 0; t < L; ++t) {
      B[(size_t)t * N + n] = sb[t];
      C[(size_t)t * N + n] = sc[t];
    }
  }
}

/* one step of the recurrence: st <- a*st + dt * x (outer) B */
static void rec_step(double *st, int P, int N, double a, double dt, const double *x, const double *B) {
  for (int p = 0; p < P; ++p) {
    double dx = dt * x[p];
    double *row = st + (size_t)p * N;
    for (int n = 0; n < N; ++n) row[n] = a * row[n] + dx * B[n];
  }
}

/* ------------------------------------------------------------------ */
/* forward                                                             */

typedef struct {
  const orc_row *r;
  const chan_set *s;
  const double *u; /* channel subset, channel-major */
  int S;
  double *y;        /* L x nh x P */
  double *final_st; /* nh x P x N */
  double *seg_in;   /* S x nh x P x N or NULL */
  double *s_ext;    /* S x nh x P x N or NULL */
  double *a_blk;    /* S x nh or NULL */
} fwd_ctx;

static void fwd_task(void *vc, int i) {
  fwd_ctx *c = (fwd_ctx *)vc;
  const orc_row *r = c->r;
  int L = r->L, P = r->P, N = r->N, S = c->S, h = c->s->h0 + i;
  int nh = c->s->h1 - c->s->h0;
  size_t PN = (size_t)P * N;
  int Ls = L / S;
  double *x = (double *)malloc(sizeof(double) * (size_t)L * P);
  double *B = (double *)malloc(sizeof(double) * (size_t)L * N);
  double *C = (double *)malloc(sizeof(double) * (size_t)L * N);
  double *st = (double *)malloc(sizeof(double) * PN);
  double *sext = (double *)malloc(sizeof(double) * PN * S);
  double *sin_ = (double *)malloc(sizeof(double) * PN * S);
  double *ablk = (double *)malloc(sizeof(double) * S);
  gather_head(r, c->s, c->u, h, x, B, C);
  double Dh = r->D[h];

  /* each segment from a zero initial state: local outputs and (S_ext, a_block) */
  for (int k = 0; k < S; ++k) {
    memset(st, 0, sizeof(double) * PN);
    double prod = 1.0;
    for (int t = k * Ls; t < (k + 1) * Ls; ++t) {
      double dt = dt_of(r, t, h);
      double a = decay_of(r, t, h, dt);
      prod *= a;
      rec_step(st, P, N, a, dt, x + (size_t)t * P, B + (size_t)t * N);
      double *yt = c->y + ((size_t)t * nh + i) * P;
      for (int p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int n = 0; n < N; ++n) acc += st[(size_t)p * N + n] * C[(size_t)t * N + n];
        yt[p] = acc + Dh * x[(size_t)t * P + p];
      }
    }
    memcpy(sext + PN * k, st, sizeof(double) * PN);
    ablk[k] = prod;
  }
  /* exclusive causal scan over the segment summaries, from the row's initial state */
  if (r->init)
    memcpy(sin_, r->init + (size_t)h * PN, sizeof(double) * PN);
  else
    memset(sin_, 0, sizeof(double) * PN);
  for (int k = 1; k < S; ++k)
    for (size_t e = 0; e < PN; ++e) sin_[PN * k + e] = ablk[k - 1] * sin_[PN * (k - 1) + e] + sext[PN * (k - 1) + e];
  double *fin = c->final_st + PN * i;
  for (size_t e = 0; e < PN; ++e) fin[e] = ablk[S - 1] * sin_[PN * (S - 1) + e] + sext[PN * (S - 1) + e];
  /* correction: carry each segment's true initial state into its outputs
   * (segment 0's is zero unless the row has an initial state) */
  for (int k = r->init ? 0 : 1; k < S; ++k) {
    const double *si = sin_ + PN * k;
    double prod = 1.0;
    for (int t = k * Ls; t < (k + 1) * Ls; ++t) {
      double dt = dt_of(r, t, h);
      prod *= decay_of(r, t, h, dt);
      double *yt = c->y + ((size_t)t * nh + i) * P;
      for (int p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int n = 0; n < N; ++n) acc += si[(size_t)p * N + n] * C[(size_t)t * N + n];
        yt[p] += prod * acc;
      }
    }
  }
  for (int k = 0; k < S; ++k) {
    if (c->seg_in) memcpy(c->seg_in + ((size_t)k * nh + i) * PN, sin_ + PN * k, sizeof(double) * PN);
    if (c->s_ext) memcpy(c->s_ext + ((size_t)k * nh + i) * PN, sext + PN * k, sizeof(double) * PN);
    if (c->a_blk) c->a_blk[(size_t)k * nh + i] = ablk[k];
  }
  free(x);
  free(B);
  free(C);
  free(st);
  free(sext);
  free(sin_);
  free(ablk);
}

/* Public: forward for heads [h0,h1) of one row, the sequence cut into S equal
 * causal segments (S=1: the plain recurrence).  Returns 0, or -1 on bad args. */
int orc_forward(const orc_row *r, int h0, int h1, int S, double *y, double *final_st, double *seg_in,
                double *s_ext, double *a_blk, int nthreads) {
  if (h0 < 0 || h1 > r->H || h0 >= h1 || S < 1 || r->L % S != 0 || r->H % r->G != 0) return -1;
  chan_set s = make_set(r, h0, h1);
  double *u = (double *)malloc(sizeof(double) * (size_t)s.nsub * r->L);
  conv_ctx cc = {r, &s, NULL, u};
  run_tasks(conv_task, &cc, s.nsub, nthreads);
  fwd_ctx c = {r, &s, u, S, y, final_st, seg_in, s_ext, a_blk};
  run_tasks(fwd_task, &c, h1 - h0, nthreads);
  free(u);
  return 0;
}

/* ------------------------------------------------------------------ */
/* backward                                                            */

typedef struct {
  const orc_row *r;
  const chan_set *s;
  const double *u;      /* channel subset, channel-major (post-conv) */
  const double *dy;     /* L x H x P (full row) */
  const double *dfinal; /* H x P x N (full row) or NULL */
  double *du_x;         /* nh x L x P */
  double *du_B;         /* nh x L x N, per-head partials */
  double *du_C;         /* nh x L x N */
  double *dinit;        /* nh x P x N: grad of the row's initial state, or NULL */
  double *ddt_raw;      /* L x nh */
  double *dA;           /* nh: dL/dA */
  double *dD;           /* nh */
} bwd_ctx;

static void bwd_task(void *vc, int i) {
  bwd_ctx *c = (bwd_ctx *)vc;
  const orc_row *r = c->r;
  int L = r->L, P = r->P, N = r->N, H = r->H, h = c->s->h0 + i;
  int nh = c->s->h1 - c->s->h0;
  size_t PN = (size_t)P * N;
  double A = -exp(r->A_log[h]), Dh = r->D[h];
  double *x = (double *)malloc(sizeof(double) * (size_t)L * P);
  double *B = (double *)malloc(sizeof(double) * (size_t)L * N);
  double *C = (double *)malloc(sizeof(double) * (size_t)L * N);
  gather_head(r, c->s, c->u, h, x, B, C);
  int nck = (L + CKPT - 1) / CKPT;
  double *ck = (double *)malloc(sizeof(double) * PN * nck);  /* state before token j*CKPT */
  double *blk = (double *)malloc(sizeof(double) * PN * CKPT); /* states h_t inside a block */
  double *st = (double *)calloc(PN, sizeof(double));
  double *G = (double *)calloc(PN, sizeof(double));
  if (r->init) memcpy(st, r->init + (size_t)h * PN, sizeof(double) * PN);
  /* forward sweep from the state before token 0, checkpointing every CKPT tokens */
  for (int t = 0; t < L; ++t) {
    if (t % CKPT == 0) memcpy(ck + PN * (t / CKPT), st, sizeof(double) * PN);
    double dt = dt_of(r, t, h);
    rec_step(st, P, N, decay_of(r, t, h, dt), dt, x + (size_t)t * P, B + (size_t)t * N);
  }
  if (c->dfinal) memcpy(G, c->dfinal + (size_t)h * PN, sizeof(double) * PN);
  double dA = 0.0, dD = 0.0;
  double *dux = c->du_x + (size_t)i * L * P;
  double *duB = c->du_B + (size_t)i * L * N;
  double *duC = c->du_C + (size_t)i * L * N;
  for (int j = nck - 1; j >= 0; --j) {
    int t0 = j * CKPT, t1 = t0 + CKPT < L ? t0 + CKPT : L;
    memcpy(st, ck + PN * j, sizeof(double) * PN);
    for (int t = t0; t < t1; ++t) {
      double dt = dt_of(r, t, h);
      rec_step(st, P, N, decay_of(r, t, h, dt), dt, x + (size_t)t * P, B + (size_t)t * N);
      memcpy(blk + PN * (t - t0), st, sizeof(double) * PN);
    }
    for (int t = t1 - 1; t >= t0; --t) {
      const double *xt = x + (size_t)t * P, *Bt = B + (size_t)t * N, *Ct = C + (size_t)t * N;
      const double *dyt = c->dy + ((size_t)t * H + h) * P;
      const double *ht = blk + PN * (t - t0);
      const double *hprev = (t == t0) ? ck + PN * j : blk + PN * (t - t0 - 1);
      double z = r->dt_raw[(size_t)t * H + h] + r->dt_bias[h];
      double dt = softplus(z);
      double a = decay_of(r, t, h, dt);
      /* G: dL/dh_t = dy_t (outer) C_t + (carried from t+1) */
      for (int p = 0; p < P; ++p)
        for (int n = 0; n < N; ++n) G[(size_t)p * N + n] += dyt[p] * Ct[n];
      double gxb = 0.0, ghp = 0.0;
      for (int p = 0; p < P; ++p) {
        double accB = 0.0;
        for (int n = 0; n < N; ++n) {
          double g = G[(size_t)p * N + n];
          accB += g * Bt[n];
          ghp += g * hprev[(size_t)p * N + n];
        }
        gxb += accB * xt[p];
        dux[(size_t)t * P + p] = dt * accB + Dh * dyt[p];
        dD += dyt[p] * xt[p];
      }
      for (int n = 0; n < N; ++n) {
        double accx = 0.0, acch = 0.0;
        for (int p = 0; p < P; ++p) {
          accx += G[(size_t)p * N + n] * xt[p];
          acch += ht[(size_t)p * N + n] * dyt[p];
        }
        duB[(size_t)t * N + n] = dt * accx;
        duC[(size_t)t * N + n] = acch;
      }
      double ddt = gxb;
      if (!is_reset(r, t)) {
        ddt += A * a * ghp;
        dA += dt * a * ghp;
      }
      c->ddt_raw[(size_t)t * nh + i] = ddt * sigmoid(z);
      /* carry to t-1 */
      for (size_t e = 0; e < PN; ++e) G[e] *= a;
    }
  }
  c->dA[i] = dA;
  c->dD[i] = dD;
  /* after the carry past token 0, G is the gradient of the state before it */
  if (c->dinit) memcpy(c->dinit + (size_t)i * PN, G, sizeof(double) * PN);
  free(x);
  free(B);
  free(C);
  free(ck);
  free(blk);
  free(st);
  free(G);
}

typedef struct {
  const orc_row *r;
  const chan_set *s;
  const double *v;  /* nsub x L pre-activation */
  const double *du; /* nsub x L grad of post-conv */
  double *dxr;      /* L x nsub grad of raw conv input (token-major) */
  double *dw;       /* nsub x 4 */
  double *db;       /* nsub */
} convb_ctx;

static void convb_task(void *vc, int j) {
  convb_ctx *c = (convb_ctx *)vc;
  const orc_row *r = c->r;
  int L = r->L, Cd = conv_dim(r), ch = set_channel(r, c->s, j), nsub = c->s->nsub;
  const double *v = c->v + (size_t)j * L, *du = c->du + (size_t)j * L;
  double *dv = (double *)malloc(sizeof(double) * (size_t)L);
  double db = 0.0, dw[DCONV] = {0, 0, 0, 0};
  for (int t = 0; t < L; ++t) {
    double sg = sigmoid(v[t]);
    dv[t] = du[t] * sg * (1.0 + v[t] * (1.0 - sg));
    db += dv[t];
  }
  for (int t = 0; t < L; ++t) {
    for (int k = 0; k < DCONV; ++k) {
      int s = t - (DCONV - 1) + k;
      if (s < 0 || !same_seq(r, s, t)) continue;
      dw[k] += dv[t] * r->xBC[(size_t)s * Cd + ch];
    }
  }
  for (int s = 0; s < L; ++s) {
    double acc = 0.0;
    for (int k = 0; k < DCONV; ++k) {
      int t = s + (DCONV - 1) - k;
      if (t >= L || !same_seq(r, s, t)) continue;
      acc += r->conv_w[(size_t)ch * DCONV + k] * dv[t];
    }
    c->dxr[(size_t)s * nsub + j] = acc;
  }
  for (int k = 0; k < DCONV; ++k) c->dw[(size_t)j * DCONV + k] = dw[k];
  c->db[j] = db;
  free(dv);
}

/* Public: backward for heads [h0,h1) of one row (the plain recurrence; the
 * segmented forward gives the same function, so its gradient is the same).
 *   dy      L x H x P  (full row)      dfinal  H x P x N (full row) or NULL
 * Outputs over the channel subset of heads [h0,h1) (x channels of those
 * heads, then B and C channels of their groups; B/C terms are summed over the
 * heads in [h0,h1) only, in head order):
 *   dxr     L x nsub      grad of the raw conv input
 *   dconv_w nsub x 4      dconv_b nsub
 * and per head:  ddt_raw L x nh,  ddt_bias nh,  dA_log nh,  dD nh, and with an
 * initial state  dinit nh x P x N  (may be NULL). */
int orc_backward(const orc_row *r, int h0, int h1, const double *dy, const double *dfinal, double *dxr,
                 double *dconv_w, double *dconv_b, double *ddt_raw, double *ddt_bias, double *dA_log,
                 double *dD, double *dinit, int nthreads) {
  if (h0 < 0 || h1 > r->H || h0 >= h1 || r->H % r->G != 0) return -1;
  chan_set s = make_set(r, h0, h1);
  int L = r->L, P = r->P, N = r->N, nh = h1 - h0;
  size_t Ls = (size_t)L;
  double *u = (double *)malloc(sizeof(double) * s.nsub * Ls);
  double *v = (double *)malloc(sizeof(double) * s.nsub * Ls);
  conv_ctx cc = {r, &s, v, u};
  run_tasks(conv_task, &cc, s.nsub, nthreads);

  double *du_x = (double *)malloc(sizeof(double) * nh * Ls * P);
  double *du_B = (double *)malloc(sizeof(double) * nh * Ls * N);
  double *du_C = (double *)malloc(sizeof(double) * nh * Ls * N);
  double *dA = (double *)malloc(sizeof(double) * nh);
  bwd_ctx bc = {r, &s, u, dy, dfinal, du_x, du_B, du_C, r->init ? dinit : NULL, ddt_raw, dA, dD};
  run_tasks(bwd_task, &bc, nh, nthreads);

  /* gradient of the post-conv channels, channel-major; B/C summed in head order */
  double *du = (double *)calloc(s.nsub * Ls, sizeof(double));
  for (int i = 0; i < nh; ++i)
    for (int p = 0; p < P; ++p)
      for (int t = 0; t < L; ++t) du[((size_t)i * P + p) * Ls + t] = du_x[((size_t)i * L + t) * P + p];
  int hpg = r->H / r->G;
  for (int i = 0; i < nh; ++i) {
    int g = (h0 + i) / hpg - s.g0;
    for (int n = 0; n < N; ++n) {
      double *dB = du + ((size_t)s.nx + (size_t)g * N + n) * Ls;
      double *dC = du + ((size_t)s.nx + (size_t)s.ng * N + (size_t)g * N + n) * Ls;
      for (int t = 0; t < L; ++t) {
        dB[t] += du_B[((size_t)i * L + t) * N + n];
        dC[t] += du_C[((size_t)i * L + t) * N + n];
      }
    }
  }
  for (int i = 0; i < nh; ++i) {
    int h = h0 + i;
    double A = -exp(r->A_log[h]);
    dA_log[i] = dA[i] * A; /* dA/dA_log = -exp(A_log) = A */
    double sacc = 0.0;
    for (int t = 0; t < L; ++t) sacc += ddt_raw[(size_t)t * nh + i];
    ddt_bias[i] = sacc;
  }
  convb_ctx cb = {r, &s, v, du, dxr, dconv_w, dconv_b};
  run_tasks(convb_task, &cb, s.nsub, nthreads);
  free(u);
  free(v);
  free(du_x);
  free(du_B);
  free(du_C);
  free(dA);
  free(du);
  return 0;
}

/* ------------------------------------------------------------------ */
/* per-sequence final states                                           */

typedef struct {
  const orc_row *r;
  const chan_set *s;
  const double *u;
  int nseq;
  double *out; /* nseq x nh x P x N */
} fin_ctx;

static void fin_task(void *vc, int i) {
  fin_ctx *c = (fin_ctx *)vc;
  const orc_row *r = c->r;
  int L = r->L, P = r->P, N = r->N, h = c->s->h0 + i, nh = c->s->h1 - c->s->h0;
  size_t PN = (size_t)P * N;
  double *x = (double *)malloc(sizeof(double) * (size_t)L * P);
  double *B = (double *)malloc(sizeof(double) * (size_t)L * N);
  double *C = (double *)malloc(sizeof(double) * (size_t)L * N);
  double *st = (double *)calloc(PN, sizeof(double));
  gather_head(r, c->s, c->u, h, x, B, C);
  if (r->init) memcpy(st, r->init + (size_t)h * PN, sizeof(double) * PN);
  int q = 0;
  for (int t = 0; t < L; ++t) {
    if (t > 0 && !same_seq(r, t - 1, t)) { /* the previous token ended a sequence */
      memcpy(c->out + ((size_t)q * nh + i) * PN, st, sizeof(double) * PN);
      ++q;
    }
    double dt = dt_of(r, t, h);
    rec_step(st, P, N, decay_of(r, t, h, dt), dt, x + (size_t)t * P, B + (size_t)t * N);
  }
  memcpy(c->out + ((size_t)q * nh + i) * PN, st, sizeof(double) * PN);
  free(x);
  free(B);
  free(C);
  free(st);
}

/* Number of packed sequences in the row (1 + the number of seq_idx changes). */
int orc_num_seqs(const orc_row *r) {
  int n = 1;
  for (int t = 1; t < r->L; ++t) n += !same_seq(r, t - 1, t);
  return n;
}

/* Public: the state after the last token of every packed sequence of the row,
 * in order, for heads [h0,h1): out is nseq x nh x P x N (the plain recurrence,
 * token by token).  Returns nseq, or -1 on bad args. */
int orc_seq_finals(const orc_row *r, int h0, int h1, double *out, int nthreads) {
  if (h0 < 0 || h1 > r->H || h0 >= h1 || r->H % r->G != 0) return -1;
  chan_set s = make_set(r, h0, h1);
  double *u = (double *)malloc(sizeof(double) * (size_t)s.nsub * r->L);
  conv_ctx cc = {r, &s, NULL, u};
  run_tasks(conv_task, &cc, s.nsub, nthreads);
  fin_ctx c = {r, &s, u, orc_num_seqs(r), out};
  run_tasks(fin_task, &c, h1 - h0, nthreads);
  free(u);
  return c.nseq;
}

/* ------------------------------------------------------------------ */
/* gated RMSNorm after the mixer core                                   */
/*
 * The Mamba2 block normalises the mixer output gated by z before its output
 * projection; the Megatron-LM PR keeps this step outside its fused function
 * ("Add state-passing context parallelism for Mamba2", description).  The
 * reading taken (Mamba2's gated RMSNorm, gate applied before the norm, one
 * norm group per B/C group of heads):
 *     g_c   = y_c * silu(z_c)
 *     r     = 1 / sqrt(mean_{c in group} g_c^2 + eps)
 *     out_c = g_c * r * w_c
 * For one row of L tokens, HP = H*P channels, G groups of HP/G channels.
 */
int orc_gated_norm_fwd(int L, int HP, int G, const double *y, const double *z, const double *w, double eps,
                       double *out) {
  if (L <= 0 || HP <= 0 || G <= 0 || HP % G != 0) return -1;
  int gs = HP / G;
  for (int t = 0; t < L; ++t)
    for (int g = 0; g < G; ++g) {
      const double *yt = y + (size_t)t * HP + (size_t)g * gs, *zt = z + (size_t)t * HP + (size_t)g * gs;
      double ss = 0.0;
      for (int c = 0; c < gs; ++c) {
        double gc = yt[c] * zt[c] * sigmoid(zt[c]);
        ss += gc * gc;
      }
      double r = 1.0 / sqrt(ss / gs + eps);
      for (int c = 0; c < gs; ++c) {
        double gc = yt[c] * zt[c] * sigmoid(zt[c]);
        out[(size_t)t * HP + (size_t)g * gs + c] = gc * r * w[(size_t)g * gs + c];
      }
    }
  return 0;
}

/* Backward of the gated RMSNorm for one row, given dout:
 *     dg_c = r w_c dout_c - g_c r^3 mean_{k in group}(w_k dout_k g_k)
 *     dy_c = dg_c silu(z_c),   dz_c = dg_c y_c silu'(z_c),
 *     dw_c += sum_t dout_c g_c r        (accumulated into dw). */
int orc_gated_norm_bwd(int L, int HP, int G, const double *y, const double *z, const double *w, double eps,
                       const double *dout, double *dy, double *dz, double *dw) {
  if (L <= 0 || HP <= 0 || G <= 0 || HP % G != 0) return -1;
  int gs = HP / G;
  for (int t = 0; t < L; ++t)
    for (int g = 0; g < G; ++g) {
      size_t o = (size_t)t * HP + (size_t)g * gs;
      double ss = 0.0, wdg = 0.0;
      for (int c = 0; c < gs; ++c) {
        double gc = y[o + c] * z[o + c] * sigmoid(z[o + c]);
        ss += gc * gc;
        wdg += w[(size_t)g * gs + c] * dout[o + c] * gc;
      }
      double r = 1.0 / sqrt(ss / gs + eps);
      double m = wdg / gs;
      for (int c = 0; c < gs; ++c) {
        double zc = z[o + c], sg = sigmoid(zc), s = zc * sg;
        double gc = y[o + c] * s;
        double dg = r * w[(size_t)g * gs + c] * dout[o + c] - gc * r * r * r * m;
        dy[o + c] = dg * s;
        dz[o + c] = dg * y[o + c] * sg * (1.0 + zc * (1.0 - sg));
        dw[(size_t)g * gs + c] += dout[o + c] * gc * r;
      }
    }
  return 0;
}
