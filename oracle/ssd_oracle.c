/*
 * Plain fp64 CPU oracle for the chunked SSD scan and the diagonal-A selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement of what the
 * GPU library computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header or constant with the CUDA library and includes
 * nothing from it.
 *
 * What it computes (the plain definition; the chunked GPU method reaches the same result up to
 * rounding order):
 *
 *   SSD recurrence, one independent problem per (batch b, head h):
 *     h_{-1}      = init_state[b,h]                        (zeros when no init is given)
 *     h_t         = exp(dA[b,t,h]) * R(theta_t) h_{t-1} + sum_r x[b,t,r,h,:] (outer) B[b,t,r,g,:]
 *     y[b,t,r,h,p]= sum_n C[b,t,r,g,n] * h_t[p,n]
 *     final[b,h]  = h_{T-1}
 *   with g = h / (H/G) the B/C group of head h.
 *   - The decay/write form is the recurrence that the serial.rs page (burn_mamba,
 *     mamba3/ssd/serial.rs) decomposes into K1..K5: K3 sums the rank-fused writes V^T B with the
 *     decay exp(cumA_last - cumA), K4 is h <- exp(da_chunk_end) h + s, and K5's MIMO mask
 *     (i//R >= j//R) means y at step t sees all R writes of step t.  V ("x" here) is pre-scaled:
 *     there is no dt factor, and no D-skip term ("No D skip is applied").
 *   - R(theta) is the optional Mamba-3 data-dependent rotation (scan.py page, steertts
 *     mamba3/scan.py, module docstring "THE TRICK" and rotate_by): it turns each interleaved
 *     pair (h[2k], h[2k+1]) of the state axis by +theta[b,t,h,k]:
 *         (a, b) -> (cos*a - sin*b, sin*a + cos*b).
 *     The oracle applies this rotation to the state directly at every step (the rotated
 *     recurrence itself), never the absorbed cumulative-angle form the GPU uses.
 *   - Rotation variants (moments.rs page, RotationSeq::Angle { rope_dim, rotate_pairwise }; the
 *     page names them without defining them, read plainly): only the first rope_dim state
 *     dimensions turn, theta then has rope_dim/2 angles per step, and the pair k is either the
 *     interleaved (2k, 2k+1) (rotate_pairwise, the default) or the split halves
 *     (k, k + rope_dim/2).
 *   - Quaternion rotation (moments.rs page, RotationSeq::Quaternion { cum_bshj4 }, given as the
 *     cumulative unit quaternion Q_t per (b, t, h) and 4-dimension block j of the state axis;
 *     named, not defined, read plainly): in place of R(theta_t), block j (dimensions 4j..4j+3,
 *     the quaternion h[4j] + h[4j+1] i + h[4j+2] j + h[4j+3] k) is multiplied on the left by
 *     the step quaternion q_t = Q_t Q_{t-1}^* (Q_{-1} = 1), so the turns up to step t compose
 *     to Q_t.  Left multiplication by a unit quaternion is orthogonal; with q = cos + i sin it
 *     turns the pairs (4j, 4j+1) and (4j+2, 4j+3) both by the angle, as R does.
 *
 *   Trapezoidal SSD (Mamba-3; scan.py page, the trapezoidal forward: the beta term carries the
 *   PREVIOUS step's write and is turned by one step less of rotation), per (b, h):
 *     S_t         = sum_r x[b,t,r,h,:] (outer) B[b,t,r,g,:]      (S_{-1} from prev_x, prev_B)
 *     h_t         = R(theta_t) (exp(dA_t) h_{t-1} + beta_t S_{t-1}) + gamma_t S_t
 *     y, final    as above.
 *   In the scan.py page's absorbed frame this is g_t = alpha_t g_{t-1} + gamma_t R(-Phi_t) S_t
 *   + beta_t R(-Phi_{t-1}) S_{t-1} with h_t = R(Phi_t) g_t; the oracle runs the physical-frame
 *   form above, state first decayed and fed the previous write, then turned, then fed the
 *   current write.
 *
 *   Selective scan (SSM Selective Scan page, problem statement), one problem per (b, d):
 *     h_{-1}[n] = 0
 *     h_t[n]    = exp(delta[b,t,d] * A[d,n]) * h_{t-1}[n] + delta[b,t,d] * B[b,t,n] * u[b,t,d]
 *     y[b,t,d]  = sum_n C[b,t,n] * h_t[n] + skip[d] * u[b,t,d]
 *
 * All arithmetic is fp64; inputs arrive as fp64 arrays (the caller upcasts the exact values the
 * GPU sees, e.g. bf16-rounded data).  Independent (b,h) or (b,d) problems are split across
 * POSIX threads; each problem is evaluated sequentially in time, so the thread count does not
 * change any result bit.
 *
 * `mutation` exists only so the test suite can show that its pins catch plausible mistakes; it
 * is 0 in every real use.  Non-zero values plant one deliberate error (see oracle_ssd_ex).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const double *x, *dA, *B, *C, *theta, *init;
  double *y, *final_state;
  int64_t batch, T, R, H, G, P, N;
  int mutation;
  int64_t nthreads;
  int64_t tid;
  /* trapezoidal form only (NULL gamma = the plain recurrence above) */
  const double *gamma, *beta, *prev_x, *prev_B;
  /* rotation variant: rope_dim (0 = N) and halves (0 = interleaved pairs) */
  int64_t rope_dim;
  int halves;
  /* quaternion rotation: cumulative unit quaternions [b, T, H, N/4, 4] (NULL = none) */
  const double* qcum;
} ssd_job;

/* Planted-mistake codes, used only by the oracle's own pin tests. */
enum {
  MUT_NONE = 0,
  MUT_NO_DECAY = 1,        /* drops the exp(dA) factor                        */
  MUT_DECAY_AFTER = 2,     /* applies the decay to the new write as well       */
  MUT_SWAP_BC = 3,         /* reads B where C belongs and C where B belongs    */
  MUT_RANK_LOCAL = 4,      /* y_{t,r} only sees the writes of ranks <= r       */
  MUT_ROT_SIGN = 5,        /* rotates by -theta instead of +theta              */
  MUT_GROUP_INDEX = 6,     /* maps head h to group h % G instead of h / (H/G)  */
  MUT_SS_NO_SKIP = 7,      /* selective scan: drops the skip term              */
  MUT_SS_DELTA_B = 8,      /* selective scan: forgets the delta factor on B    */
  MUT_TRAP_NO_BETA = 9,    /* trapezoidal: drops the beta (previous-write) term */
  MUT_TRAP_BETA_TURNED_LATE = 10, /* trapezoidal: feeds beta*S_{t-1} after the turn */
  MUT_TRAP_BETA_CURRENT = 11,     /* trapezoidal: beta multiplies S_t, not S_{t-1} */
  MUT_ROT_INTERLEAVED = 12,       /* rotation variant: ignores the split-halves pairing */
  MUT_ROPE_LAST_DIMS = 13,        /* rotation variant: turns the last rope_dim dims */
  MUT_QUAT_RIGHT = 20,            /* quaternion: multiplies on the right, not the left */
  MUT_QUAT_CUM_AS_STEP = 21,      /* quaternion: turns by Q_t instead of Q_t Q_{t-1}^* */
};

/* Hamilton product o = a b of quaternions stored (w, x, y, z) = w + x i + y j + z k. */
static void quat_mul(const double* a, const double* b, double* o) {
  const double w = a[0] * b[0] - a[1] * b[1] - a[2] * b[2] - a[3] * b[3];
  const double x = a[0] * b[1] + a[1] * b[0] + a[2] * b[3] - a[3] * b[2];
  const double y = a[0] * b[2] - a[1] * b[3] + a[2] * b[0] + a[3] * b[1];
  const double z = a[0] * b[3] + a[1] * b[2] - a[2] * b[1] + a[3] * b[0];
  o[0] = w;
  o[1] = x;
  o[2] = y;
  o[3] = z;
}

/* Quaternion rotation of one step (moments.rs page, RotationSeq::Quaternion { cum_bshj4 }):
 * block k of the state axis, dimensions (4k .. 4k+3) read as the quaternion
 * h[4k] + h[4k+1] i + h[4k+2] j + h[4k+3] k, is turned by LEFT multiplication with the step's
 * unit quaternion q_t = Q_t Q_{t-1}^* (Q the given cumulative quaternions, Q_{-1} = 1), so that
 * the turns compose to Q_t over steps 0..t. */
static void quat_turn_state(const ssd_job* j, int64_t b, int64_t hh, int64_t t, double* h) {
  const int64_t T = j->T, H = j->H, P = j->P, N = j->N, K = N / 4;
  const double* Qt = j->qcum + ((b * T + t) * H + hh) * K * 4;
  const double* Qp = t > 0 ? j->qcum + ((b * T + t - 1) * H + hh) * K * 4 : NULL;
  for (int64_t k = 0; k < K; ++k) {
    double q[4];
    if (j->mutation == MUT_QUAT_CUM_AS_STEP || !Qp) {
      memcpy(q, Qt + 4 * k, sizeof(q));
    } else {
      const double conj[4] = {Qp[4 * k], -Qp[4 * k + 1], -Qp[4 * k + 2], -Qp[4 * k + 3]};
      quat_mul(Qt + 4 * k, conj, q);
    }
    for (int64_t p = 0; p < P; ++p) {
      double* v = h + p * N + 4 * k;
      double o[4];
      if (j->mutation == MUT_QUAT_RIGHT) {
        quat_mul(v, q, o);
      } else {
        quat_mul(q, v, o);
      }
      memcpy(v, o, sizeof(o));
    }
  }
}

/* The pair of state dimensions that angle k of the rotation variant turns. */
static void rot_pair(const ssd_job* j, int64_t k, int64_t* d0, int64_t* d1) {
  const int64_t rd = j->rope_dim > 0 ? j->rope_dim : j->N;
  const int64_t off = (j->mutation == MUT_ROPE_LAST_DIMS) ? j->N - rd : 0;
  if (j->halves && j->mutation != MUT_ROT_INTERLEAVED) {
    *d0 = off + k;
    *d1 = off + k + rd / 2;
  } else {
    *d0 = off + 2 * k;
    *d1 = off + 2 * k + 1;
  }
}

/* The trapezoidal recurrence for one (b, h); h and the two write buffers hold P*N doubles. */
static void trap_one(const ssd_job* j, int64_t b, int64_t hh, double* h, double* sprev,
                     double* scur) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N;
  const int64_t g = hh / (H / G);
  if (j->init) {
    memcpy(h, j->init + ((b * H + hh) * P) * N, sizeof(double) * P * N);
  } else {
    memset(h, 0, sizeof(double) * P * N);
  }
  /* S_{-1}: the write of the step before the first (the previous call's last step) */
  for (int64_t p = 0; p < P; ++p) {
    for (int64_t n = 0; n < N; ++n) {
      double w = 0.0;
      if (j->prev_x && j->prev_B) {
        for (int64_t r = 0; r < R; ++r)
          w += j->prev_x[((b * R + r) * H + hh) * P + p] * j->prev_B[((b * R + r) * G + g) * N + n];
      }
      sprev[p * N + n] = w;
    }
  }
  for (int64_t t = 0; t < T; ++t) {
    const double a = exp(j->dA[(b * T + t) * H + hh]);
    const double gm = j->gamma[(b * T + t) * H + hh];
    const double bt = j->beta[(b * T + t) * H + hh];
    for (int64_t p = 0; p < P; ++p) {
      for (int64_t n = 0; n < N; ++n) {
        double w = 0.0;
        for (int64_t r = 0; r < R; ++r)
          w += j->x[(((b * T + t) * R + r) * H + hh) * P + p] *
               j->B[(((b * T + t) * R + r) * G + g) * N + n];
        scur[p * N + n] = w;
      }
    }
    const double* fed = (j->mutation == MUT_TRAP_BETA_CURRENT) ? scur : sprev;
    const int late = j->mutation == MUT_TRAP_BETA_TURNED_LATE;
    const double bw = (j->mutation == MUT_TRAP_NO_BETA) ? 0.0 : bt;
    for (int64_t e = 0; e < P * N; ++e) h[e] = a * h[e] + (late ? 0.0 : bw * fed[e]);
    if (j->theta) {
      const double* th = j->theta + ((b * T + t) * H + hh) * (N / 2);
      for (int64_t k = 0; k < N / 2; ++k) {
        const double c = cos(th[k]), s = sin(th[k]);
        for (int64_t p = 0; p < P; ++p) {
          double* hp = h + p * N;
          const double e0 = hp[2 * k], o0 = hp[2 * k + 1];
          hp[2 * k] = c * e0 - s * o0;
          hp[2 * k + 1] = s * e0 + c * o0;
        }
      }
    }
    for (int64_t e = 0; e < P * N; ++e) h[e] += gm * scur[e] + (late ? bw * fed[e] : 0.0);
    for (int64_t r = 0; r < R; ++r) {
      const double* cv = j->C + (((b * T + t) * R + r) * G + g) * N;
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += cv[n] * h[p * N + n];
        j->y[(((b * T + t) * R + r) * H + hh) * P + p] = acc;
      }
    }
    memcpy(sprev, scur, sizeof(double) * P * N);
  }
  if (j->final_state) {
    memcpy(j->final_state + ((b * H + hh) * P) * N, h, sizeof(double) * P * N);
  }
}

static void ssd_one(const ssd_job* j, int64_t b, int64_t hh, double* h) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N;
  const int64_t heads_per_group = H / G;
  const int64_t g = (j->mutation == MUT_GROUP_INDEX) ? (hh % G) : (hh / heads_per_group);
  const double* Bsrc = (j->mutation == MUT_SWAP_BC) ? j->C : j->B;
  const double* Csrc = (j->mutation == MUT_SWAP_BC) ? j->B : j->C;

  if (j->init) {
    memcpy(h, j->init + ((b * H + hh) * P) * N, sizeof(double) * P * N);
  } else {
    memset(h, 0, sizeof(double) * P * N);
  }
  for (int64_t t = 0; t < T; ++t) {
    const double a = (j->mutation == MUT_NO_DECAY) ? 1.0 : exp(j->dA[(b * T + t) * H + hh]);
    if (j->qcum) quat_turn_state(j, b, hh, t, h);
    if (j->theta) {
      const int64_t K = (j->rope_dim > 0 ? j->rope_dim : N) / 2;
      const double* th = j->theta + ((b * T + t) * H + hh) * K;
      for (int64_t k = 0; k < K; ++k) {
        const double ang = (j->mutation == MUT_ROT_SIGN) ? -th[k] : th[k];
        const double c = cos(ang), s = sin(ang);
        int64_t d0, d1;
        rot_pair(j, k, &d0, &d1);
        for (int64_t p = 0; p < P; ++p) {
          double* hp = h + p * N;
          const double e = hp[d0], o = hp[d1];
          hp[d0] = c * e - s * o;
          hp[d1] = s * e + c * o;
        }
      }
    }
    for (int64_t p = 0; p < P; ++p) {
      for (int64_t n = 0; n < N; ++n) {
        double w = 0.0;
        for (int64_t r = 0; r < R; ++r) {
          const double xv = j->x[(((b * T + t) * R + r) * H + hh) * P + p];
          const double bv = Bsrc[(((b * T + t) * R + r) * G + g) * N + n];
          w += xv * bv;
        }
        if (j->mutation == MUT_DECAY_AFTER) {
          h[p * N + n] = a * (h[p * N + n] + w);
        } else {
          h[p * N + n] = a * h[p * N + n] + w;
        }
      }
    }
    for (int64_t r = 0; r < R; ++r) {
      const double* cv = Csrc + (((b * T + t) * R + r) * G + g) * N;
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        if (j->mutation == MUT_RANK_LOCAL) {
          /* Recompute the state as if only ranks 0..r had written at step t. */
          for (int64_t n = 0; n < N; ++n) {
            double hv = h[p * N + n];
            for (int64_t r2 = r + 1; r2 < R; ++r2) {
              hv -= j->x[(((b * T + t) * R + r2) * H + hh) * P + p] *
                    Bsrc[(((b * T + t) * R + r2) * G + g) * N + n];
            }
            acc += cv[n] * hv;
          }
        } else {
          for (int64_t n = 0; n < N; ++n) acc += cv[n] * h[p * N + n];
        }
        j->y[(((b * T + t) * R + r) * H + hh) * P + p] = acc;
      }
    }
  }
  if (j->final_state) {
    memcpy(j->final_state + ((b * H + hh) * P) * N, h, sizeof(double) * P * N);
  }
}

static void* ssd_worker(void* arg) {
  const ssd_job* j = (const ssd_job*)arg;
  double* h = (double*)malloc(sizeof(double) * j->P * j->N * 3);
  if (!h) return (void*)1;
  for (int64_t idx = j->tid; idx < j->batch * j->H; idx += j->nthreads) {
    if (j->gamma) {
      trap_one(j, idx / j->H, idx % j->H, h, h + j->P * j->N, h + 2 * j->P * j->N);
    } else {
      ssd_one(j, idx / j->H, idx % j->H, h);
    }
  }
  free(h);
  return NULL;
}

static int64_t clamp_threads(int64_t nthreads, int64_t work) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > work) nthreads = work;
  if (nthreads > 512) nthreads = 512;
  return nthreads < 1 ? 1 : nthreads;
}

static int run_ssd(const double* x, const double* dA, const double* B, const double* C,
                   const double* theta, const double* init_state, double* y, double* final_state,
                   int64_t batch, int64_t T, int64_t R, int64_t H, int64_t G, int64_t P, int64_t N,
                   int64_t nthreads, int mutation, const double* gamma, const double* beta,
                   const double* prev_x, const double* prev_B, int64_t rope_dim, int halves,
                   const double* qcum) {
  if (!x || !dA || !B || !C || !y) return -1;
  if (qcum && ((N % 4) != 0 || theta)) return -7;
  if (batch < 0 || T < 0 || R < 1 || H < 1 || G < 1 || P < 1 || N < 1) return -2;
  if (H % G != 0) return -3;
  if (theta && (N % 2 != 0)) return -4;
  if (rope_dim < 0 || rope_dim > N || (rope_dim % 2) != 0) return -6;
  if (batch == 0 || T == 0) {
    if (final_state) {
      for (int64_t i = 0; i < batch * H * P * N; ++i)
        final_state[i] = init_state ? init_state[i] : 0.0;
    }
    return 0;
  }
  const int64_t nt = clamp_threads(nthreads, batch * H);
  ssd_job* jobs = (ssd_job*)calloc((size_t)nt, sizeof(ssd_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -5;
  }
  int rc = 0;
  for (int64_t i = 0; i < nt; ++i) {
    ssd_job j = {x,  dA, B,    C,     theta,  init_state, y,      final_state, batch, T,
                 R,  H,  G,    P,     N,      mutation,   nt,     i,           gamma, beta,
                 prev_x, prev_B, rope_dim, halves, qcum};
    jobs[i] = j;
  }
  for (int64_t i = 1; i < nt; ++i) pthread_create(&th[i], NULL, ssd_worker, &jobs[i]);
  if (ssd_worker(&jobs[0]) != NULL) rc = -5;
  for (int64_t i = 1; i < nt; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret != NULL) rc = -5;
  }
  free(jobs);
  free(th);
  return rc;
}

/* Returns 0 on success, a negative value on invalid arguments or allocation failure. */
int oracle_ssd_ex(const double* x, const double* dA, const double* B, const double* C,
                  const double* theta, const double* init_state, double* y, double* final_state,
                  int64_t batch, int64_t T, int64_t R, int64_t H, int64_t G, int64_t P, int64_t N,
                  int64_t nthreads, int mutation) {
  return run_ssd(x, dA, B, C, theta, init_state, y, final_state, batch, T, R, H, G, P, N,
                 nthreads, mutation, NULL, NULL, NULL, NULL, 0, 0, NULL);
}

/* Rotation variants: theta [b,T,H,rope_dim/2] (rope_dim 0 = dstate); halves = 1 pairs the
 * dimensions (k, k + rope_dim/2) instead of (2k, 2k+1). */
int oracle_ssd_rot_ex(const double* x, const double* dA, const double* B, const double* C,
                      const double* theta, const double* init_state, double* y,
                      double* final_state, int64_t batch, int64_t T, int64_t R, int64_t H,
                      int64_t G, int64_t P, int64_t N, int64_t rope_dim, int halves,
                      int64_t nthreads, int mutation) {
  return run_ssd(x, dA, B, C, theta, init_state, y, final_state, batch, T, R, H, G, P, N,
                 nthreads, mutation, NULL, NULL, NULL, NULL, rope_dim, halves, NULL);
}

/* Quaternion rotation: qcum [b,T,H,N/4,4] cumulative unit quaternions (w, x, y, z); N % 4 == 0,
 * no theta.  Block k of the state is turned by left multiplication with Q_t Q_{t-1}^* at step t. */
int oracle_ssd_quat_ex(const double* x, const double* dA, const double* B, const double* C,
                       const double* qcum, const double* init_state, double* y,
                       double* final_state, int64_t batch, int64_t T, int64_t R, int64_t H,
                       int64_t G, int64_t P, int64_t N, int64_t nthreads, int mutation) {
  if (!qcum) return -1;
  return run_ssd(x, dA, B, C, NULL, init_state, y, final_state, batch, T, R, H, G, P, N,
                 nthreads, mutation, NULL, NULL, NULL, NULL, 0, 0, qcum);
}

/* Trapezoidal form: gamma, beta [b,T,H]; prev_x [b,R,H,P] and prev_B [b,R,G,N] may be NULL
 * (no previous write). */
int oracle_ssd_trap_ex(const double* x, const double* dA, const double* B, const double* C,
                       const double* gamma, const double* beta, const double* theta,
                       const double* init_state, const double* prev_x, const double* prev_B,
                       double* y, double* final_state, int64_t batch, int64_t T, int64_t R,
                       int64_t H, int64_t G, int64_t P, int64_t N, int64_t nthreads, int mutation) {
  if (!gamma || !beta) return -1;
  return run_ssd(x, dA, B, C, theta, init_state, y, final_state, batch, T, R, H, G, P, N,
                 nthreads, mutation, gamma, beta, prev_x, prev_B, 0, 0, NULL);
}

int oracle_ssd(const double* x, const double* dA, const double* B, const double* C,
               const double* theta, const double* init_state, double* y, double* final_state,
               int64_t batch, int64_t T, int64_t R, int64_t H, int64_t G, int64_t P, int64_t N,
               int64_t nthreads) {
  return oracle_ssd_ex(x, dA, B, C, theta, init_state, y, final_state, batch, T, R, H, G, P, N,
                       nthreads, MUT_NONE);
}

/* ---------------------------------------------------------------------------------------- */
/* Backward of the (unrotated) SSD recurrence                                                */
/* ---------------------------------------------------------------------------------------- */
/*
 * Reverse mode of h_t = exp(dA_t) R(theta_t) h_{t-1} + sum_r x_{t,r} (outer) B_{t,r},
 * y_{t,r} = C_{t,r} . h_t (R(theta) = I when theta is NULL; interleaved pairs, all of dstate)
 * for the loss <dy, y> + <dfinal, h_{T-1}> (the backward the scan.py page asks a trainable scan
 * to have), per (b, h), walking t from T-1 down with g = dL/dh_t and u_t = R(theta_t) h_{t-1}:
 *   g   += sum_r dy_{t,r} (outer) C_{t,r}            dC_{t,r} += h_t^T dy_{t,r}
 *   dx_{t,r} = g B_{t,r}     dB_{t,r} += g^T x_{t,r}   ddA_t = exp(dA_t) <g, u_t>
 *   dtheta_{t,k} = exp(dA_t) sum_p (g[p,2k+1] u_t[p,2k] - g[p,2k] u_t[p,2k+1])
 *                  (the derivative of the turn of pair k is the quarter turn J u)
 *   g   <- exp(dA_t) R(theta_t)^T g = exp(dA_t) R(-theta_t) g;   dinit = g after t = 0.
 * dB and dC sum over the heads of a group.  States are recomputed forward from checkpoints every
 * kCkpt steps, so memory stays O((T / kCkpt + kCkpt) P N) per problem.
 */
enum { MUT_BWD_DY_AFTER_DECAY = 14, MUT_BWD_NO_DECAY_IN_DDA = 15, MUT_BWD_TURN_FORWARD = 16 };

typedef struct {
  const double *x, *dA, *B, *C, *theta, *init, *dy, *dfinal;
  double *dx, *ddA, *dB, *dC, *dtheta, *dinit;
  int64_t batch, T, R, H, G, P, N;
  int mutation;
  int64_t nthreads, tid;
  pthread_mutex_t* lock;   /* dB/dC are shared by the heads of a group */
} bwd_job;

#define ORACLE_CKPT 64

/* Turns every interleaved pair (2k, 2k+1) of each of the P rows of v (P x N) by sign * th[k]. */
static void bwd_turn(const double* th, int64_t P, int64_t N, double sign, double* v) {
  for (int64_t k = 0; k < N / 2; ++k) {
    const double c = cos(sign * th[k]), s = sin(sign * th[k]);
    for (int64_t p = 0; p < P; ++p) {
      double* vp = v + p * N;
      const double e = vp[2 * k], o = vp[2 * k + 1];
      vp[2 * k] = c * e - s * o;
      vp[2 * k + 1] = s * e + c * o;
    }
  }
}

/* One step of the forward recurrence: hn = exp(dA_t) R(theta_t) hp + sum_r x_{t,r} B_{t,r}. */
static void bwd_forward_step(const bwd_job* j, int64_t b, int64_t hh, int64_t g_, int64_t t,
                             const double* hp, double* hn) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N;
  const double a = exp(j->dA[(b * T + t) * H + hh]);
  memcpy(hn, hp, sizeof(double) * P * N);
  if (j->theta) bwd_turn(j->theta + ((b * T + t) * H + hh) * (N / 2), P, N, 1.0, hn);
  for (int64_t p = 0; p < P; ++p)
    for (int64_t n = 0; n < N; ++n) {
      double w = 0.0;
      for (int64_t r = 0; r < R; ++r)
        w += j->x[(((b * T + t) * R + r) * H + hh) * P + p] *
             j->B[(((b * T + t) * R + r) * G + g_) * N + n];
      hn[p * N + n] = a * hn[p * N + n] + w;
    }
}

static void bwd_one(const bwd_job* j, int64_t b, int64_t hh, double* ck, double* seg, double* g,
                    double* u, double* dBl, double* dCl) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N, PN = P * N;
  const int64_t g_ = hh / (H / G);
  const int64_t nck = (T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  /* forward pass keeping the state entering every checkpoint segment */
  double* h = seg;   /* rows 0 and 1 of seg as the running state */
  if (j->init) {
    memcpy(h, j->init + ((b * H + hh) * P) * N, sizeof(double) * PN);
  } else {
    memset(h, 0, sizeof(double) * PN);
  }
  for (int64_t t = 0; t < T; ++t) {
    if (t % ORACLE_CKPT == 0) memcpy(ck + (t / ORACLE_CKPT) * PN, h, sizeof(double) * PN);
    bwd_forward_step(j, b, hh, g_, t, h, seg + PN);
    memcpy(h, seg + PN, sizeof(double) * PN);
  }
  if (j->dfinal) {
    memcpy(g, j->dfinal + ((b * H + hh) * P) * N, sizeof(double) * PN);
  } else {
    memset(g, 0, sizeof(double) * PN);
  }
  memset(dBl, 0, sizeof(double) * T * R * N);
  memset(dCl, 0, sizeof(double) * T * R * N);
  for (int64_t c = nck - 1; c >= 0; --c) {
    const int64_t t0 = c * ORACLE_CKPT, t1 = (t0 + ORACLE_CKPT < T) ? t0 + ORACLE_CKPT : T;
    /* recompute the states h_{t0-1} .. h_{t1-1} into seg rows 0 .. (t1 - t0) */
    memcpy(seg, ck + c * PN, sizeof(double) * PN);
    for (int64_t t = t0; t < t1; ++t)
      bwd_forward_step(j, b, hh, g_, t, seg + (t - t0) * PN, seg + (t - t0 + 1) * PN);
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double a = exp(j->dA[(b * T + t) * H + hh]);
      const double* th = j->theta ? j->theta + ((b * T + t) * H + hh) * (N / 2) : NULL;
      const double* ht = seg + (t - t0 + 1) * PN;   /* h_t */
      const double* hprev = seg + (t - t0) * PN;    /* h_{t-1} */
      for (int64_t r = 0; r < R; ++r) {
        const double* dyv = j->dy + (((b * T + t) * R + r) * H + hh) * P;
        const double* cv = j->C + (((b * T + t) * R + r) * G + g_) * N;
        for (int64_t n = 0; n < N; ++n) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p) s += dyv[p] * ht[p * N + n];
          dCl[(t * R + r) * N + n] += s;
        }
        if (j->mutation != MUT_BWD_DY_AFTER_DECAY)
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) g[p * N + n] += dyv[p] * cv[n];
      }
      for (int64_t r = 0; r < R; ++r) {
        const double* xv = j->x + (((b * T + t) * R + r) * H + hh) * P;
        const double* bv = j->B + (((b * T + t) * R + r) * G + g_) * N;
        for (int64_t p = 0; p < P; ++p) {
          double s = 0.0;
          for (int64_t n = 0; n < N; ++n) s += g[p * N + n] * bv[n];
          j->dx[(((b * T + t) * R + r) * H + hh) * P + p] = s;
        }
        for (int64_t n = 0; n < N; ++n) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p) s += g[p * N + n] * xv[p];
          dBl[(t * R + r) * N + n] += s;
        }
      }
      /* u_t = R(theta_t) h_{t-1}, the state the decay multiplies */
      memcpy(u, hprev, sizeof(double) * PN);
      if (th) bwd_turn(th, P, N, 1.0, u);
      double da = 0.0;
      for (int64_t e = 0; e < PN; ++e) da += g[e] * u[e];
      j->ddA[(b * T + t) * H + hh] = (j->mutation == MUT_BWD_NO_DECAY_IN_DDA) ? da : a * da;
      if (th && j->dtheta) {
        double* dth = j->dtheta + ((b * T + t) * H + hh) * (N / 2);
        for (int64_t k = 0; k < N / 2; ++k) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p)
            s += g[p * N + 2 * k + 1] * u[p * N + 2 * k] - g[p * N + 2 * k] * u[p * N + 2 * k + 1];
          dth[k] = a * s;
        }
      }
      for (int64_t e = 0; e < PN; ++e) g[e] *= a;
      if (th) bwd_turn(th, P, N, (j->mutation == MUT_BWD_TURN_FORWARD) ? 1.0 : -1.0, g);
      if (j->mutation == MUT_BWD_DY_AFTER_DECAY) {   /* the planted mistake: dy lands late */
        for (int64_t r = 0; r < R; ++r) {
          const double* dyv = j->dy + (((b * T + t) * R + r) * H + hh) * P;
          const double* cv = j->C + (((b * T + t) * R + r) * G + g_) * N;
          for (int64_t p = 0; p < P; ++p)
            for (int64_t n = 0; n < N; ++n) g[p * N + n] += dyv[p] * cv[n];
        }
      }
    }
  }
  if (j->dinit) memcpy(j->dinit + ((b * H + hh) * P) * N, g, sizeof(double) * PN);
  pthread_mutex_lock(j->lock);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t n = 0; n < N; ++n) {
        const int64_t o = (((b * T + t) * R + r) * G + g_) * N + n;
        j->dB[o] += dBl[(t * R + r) * N + n];
        j->dC[o] += dCl[(t * R + r) * N + n];
      }
  pthread_mutex_unlock(j->lock);
}

static void* bwd_worker(void* arg) {
  const bwd_job* j = (const bwd_job*)arg;
  const int64_t PN = j->P * j->N, nck = (j->T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  double* ck = (double*)malloc(sizeof(double) * PN * (size_t)nck);
  double* seg = (double*)malloc(sizeof(double) * PN * (ORACLE_CKPT + 1));
  double* g = (double*)malloc(sizeof(double) * PN);
  double* u = (double*)malloc(sizeof(double) * PN);
  double* dBl = (double*)malloc(sizeof(double) * j->T * j->R * j->N);
  double* dCl = (double*)malloc(sizeof(double) * j->T * j->R * j->N);
  void* rc = NULL;
  if (!ck || !seg || !g || !u || !dBl || !dCl) {
    rc = (void*)1;
  } else {
    for (int64_t idx = j->tid; idx < j->batch * j->H; idx += j->nthreads)
      bwd_one(j, idx / j->H, idx % j->H, ck, seg, g, u, dBl, dCl);
  }
  free(ck);
  free(seg);
  free(g);
  free(u);
  free(dBl);
  free(dCl);
  return rc;
}

/* Backward of the SSD (rotated when theta [b,T,H,N/2] is given): dy [b,T,R,H,P] and dfinal
 * [b,H,P,N] (nullable) in; dx, ddA, dB, dC (zeroed here), dtheta (nullable; needs theta) and
 * dinit (nullable) out.  Returns 0 or a negative error. */
int oracle_ssd_backward_ex(const double* x, const double* dA, const double* B, const double* C,
                           const double* theta, const double* init_state, const double* dy,
                           const double* dfinal, double* dx, double* ddA, double* dB, double* dC,
                           double* dtheta, double* dinit, int64_t batch, int64_t T, int64_t R,
                           int64_t H, int64_t G, int64_t P, int64_t N, int64_t nthreads,
                           int mutation) {
  if (!x || !dA || !B || !C || !dy || !dx || !ddA || !dB || !dC) return -1;
  if (batch < 1 || T < 1 || R < 1 || H < 1 || G < 1 || P < 1 || N < 1) return -2;
  if (H % G != 0) return -3;
  if (theta && (N % 2) != 0) return -4;
  memset(dB, 0, sizeof(double) * (size_t)(batch * T * R * G * N));
  memset(dC, 0, sizeof(double) * (size_t)(batch * T * R * G * N));
  const int64_t nt = clamp_threads(nthreads, batch * H);
  bwd_job* jobs = (bwd_job*)calloc((size_t)nt, sizeof(bwd_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  pthread_mutex_t lock;
  if (!jobs || !th || pthread_mutex_init(&lock, NULL) != 0) {
    free(jobs);
    free(th);
    return -5;
  }
  for (int64_t i = 0; i < nt; ++i) {
    bwd_job jb = {x,   dA,  B,  C,  theta,  init_state, dy,    dfinal, dx, ddA, dB, dC,
                  dtheta, dinit, batch, T, R, H, G, P, N, mutation, nt, i, &lock};
    jobs[i] = jb;
  }
  int rc = 0;
  for (int64_t i = 1; i < nt; ++i) pthread_create(&th[i], NULL, bwd_worker, &jobs[i]);
  if (bwd_worker(&jobs[0]) != NULL) rc = -5;
  for (int64_t i = 1; i < nt; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret != NULL) rc = -5;
  }
  pthread_mutex_destroy(&lock);
  free(jobs);
  free(th);
  return rc;
}

/* ---------------------------------------------------------------------------------------- */
/* Backward of the trapezoidal SSD recurrence                                                */
/* ---------------------------------------------------------------------------------------- */
/*
 * Reverse mode of the trapezoidal recurrence (scan.py page, the trapezoidal forward; the forward
 * is trap_one above), per (b, h), with S_t = sum_r x_{t,r} (outer) B_{t,r} (S_{-1} the previous
 * write), u_t = exp(dA_t) h_{t-1} + beta_t S_{t-1}, v_t = R(theta_t) u_t, h_t = v_t + gamma_t S_t,
 * for the loss <dy, y> + <dfinal, h_{T-1}>.  Walking t from T-1 down with g = dL/dh_t and
 * dS = dL/dS_t (which already holds beta_{t+1} du_{t+1} from the step after):
 *   g  += sum_r dy_{t,r} (outer) C_{t,r}            dC_{t,r} += h_t^T dy_{t,r}
 *   dS += gamma_t g;  dgamma_t = <g, S_t>;  dx_{t,r} = dS B_{t,r};  dB_{t,r} += dS^T x_{t,r}
 *   dtheta_{t,k} = sum_p (g[p,2k+1] v_t[p,2k] - g[p,2k] v_t[p,2k+1])
 *   du = R(-theta_t) g;  ddA_t = exp(dA_t) <du, h_{t-1}>;  dbeta_t = <du, S_{t-1}>
 *   dS <- beta_t du (for S_{t-1});  g <- exp(dA_t) du
 * and after t = 0: dinit = g, dprev_x_r = dS prev_B_r, dprev_B_r = dS^T prev_x_r.  dB, dC and
 * dprev_B sum over the heads of a group.  States are recomputed from checkpoints every kCkpt
 * steps.
 */
enum { MUT_TBWD_NO_BETA_CARRY = 17 };

typedef struct {
  const double *x, *dA, *B, *C, *gamma, *beta, *theta, *init, *prev_x, *prev_B, *dy, *dfinal;
  double *dx, *ddA, *dB, *dC, *dgamma, *dbeta, *dtheta, *dinit, *dprev_x, *dprev_B;
  int64_t batch, T, R, H, G, P, N;
  int mutation;
  int64_t nthreads, tid;
  pthread_mutex_t* lock;
} tbwd_job;

/* S = sum_r x_r (outer) B_r of step t (t = -1: the previous write, zero when absent). */
static void tbwd_write(const tbwd_job* j, int64_t b, int64_t hh, int64_t g_, int64_t t,
                       double* S) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N;
  for (int64_t p = 0; p < P; ++p)
    for (int64_t n = 0; n < N; ++n) {
      double w = 0.0;
      for (int64_t r = 0; r < R; ++r) {
        if (t >= 0) {
          w += j->x[(((b * T + t) * R + r) * H + hh) * P + p] *
               j->B[(((b * T + t) * R + r) * G + g_) * N + n];
        } else if (j->prev_x) {
          w += j->prev_x[((b * R + r) * H + hh) * P + p] * j->prev_B[((b * R + r) * G + g_) * N + n];
        }
      }
      S[p * N + n] = w;
    }
}

/* One forward step: from h_{t-1} (hp) to u_t, v_t and h_t (hn); Sp = S_{t-1}, Sc = S_t. */
static void tbwd_step(const tbwd_job* j, int64_t b, int64_t hh, int64_t t, const double* hp,
                      const double* Sp, const double* Sc, double* u, double* v, double* hn) {
  const int64_t T = j->T, H = j->H, P = j->P, N = j->N, PN = P * N;
  const double a = exp(j->dA[(b * T + t) * H + hh]);
  const double bt = j->beta[(b * T + t) * H + hh], gm = j->gamma[(b * T + t) * H + hh];
  for (int64_t e = 0; e < PN; ++e) u[e] = a * hp[e] + bt * Sp[e];
  memcpy(v, u, sizeof(double) * PN);
  if (j->theta) bwd_turn(j->theta + ((b * T + t) * H + hh) * (N / 2), P, N, 1.0, v);
  for (int64_t e = 0; e < PN; ++e) hn[e] = v[e] + gm * Sc[e];
}

static void tbwd_one(const tbwd_job* j, int64_t b, int64_t hh, double* ck, double* seg,
                     double* g, double* dS, double* Sp, double* Sc, double* u, double* v,
                     double* tmp, double* dBl, double* dCl, double* dpB) {
  const int64_t T = j->T, R = j->R, H = j->H, G = j->G, P = j->P, N = j->N, PN = P * N;
  const int64_t g_ = hh / (H / G);
  const int64_t nck = (T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  double* h = seg;
  if (j->init) {
    memcpy(h, j->init + ((b * H + hh) * P) * N, sizeof(double) * PN);
  } else {
    memset(h, 0, sizeof(double) * PN);
  }
  for (int64_t t = 0; t < T; ++t) {
    if (t % ORACLE_CKPT == 0) memcpy(ck + (t / ORACLE_CKPT) * PN, h, sizeof(double) * PN);
    tbwd_write(j, b, hh, g_, t - 1, Sp);
    tbwd_write(j, b, hh, g_, t, Sc);
    tbwd_step(j, b, hh, t, h, Sp, Sc, u, v, tmp);
    memcpy(h, tmp, sizeof(double) * PN);
  }
  if (j->dfinal) {
    memcpy(g, j->dfinal + ((b * H + hh) * P) * N, sizeof(double) * PN);
  } else {
    memset(g, 0, sizeof(double) * PN);
  }
  memset(dS, 0, sizeof(double) * PN);
  memset(dBl, 0, sizeof(double) * T * R * N);
  memset(dCl, 0, sizeof(double) * T * R * N);
  for (int64_t c = nck - 1; c >= 0; --c) {
    const int64_t t0 = c * ORACLE_CKPT, t1 = (t0 + ORACLE_CKPT < T) ? t0 + ORACLE_CKPT : T;
    memcpy(seg, ck + c * PN, sizeof(double) * PN);
    for (int64_t t = t0; t < t1; ++t) {   /* h_{t0-1} .. h_{t1-1} into seg rows 0 .. t1-t0 */
      tbwd_write(j, b, hh, g_, t - 1, Sp);
      tbwd_write(j, b, hh, g_, t, Sc);
      tbwd_step(j, b, hh, t, seg + (t - t0) * PN, Sp, Sc, u, v, seg + (t - t0 + 1) * PN);
    }
    for (int64_t t = t1 - 1; t >= t0; --t) {
      const double a = exp(j->dA[(b * T + t) * H + hh]);
      const double bt = j->beta[(b * T + t) * H + hh], gm = j->gamma[(b * T + t) * H + hh];
      const double* ht = seg + (t - t0 + 1) * PN;
      const double* hprev = seg + (t - t0) * PN;
      tbwd_write(j, b, hh, g_, t - 1, Sp);
      tbwd_write(j, b, hh, g_, t, Sc);
      tbwd_step(j, b, hh, t, hprev, Sp, Sc, u, v, tmp);
      for (int64_t r = 0; r < R; ++r) {
        const double* dyv = j->dy + (((b * T + t) * R + r) * H + hh) * P;
        const double* cv = j->C + (((b * T + t) * R + r) * G + g_) * N;
        for (int64_t n = 0; n < N; ++n) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p) s += dyv[p] * ht[p * N + n];
          dCl[(t * R + r) * N + n] += s;
        }
        for (int64_t p = 0; p < P; ++p)
          for (int64_t n = 0; n < N; ++n) g[p * N + n] += dyv[p] * cv[n];
      }
      double dgm = 0.0;
      for (int64_t e = 0; e < PN; ++e) {
        dS[e] += gm * g[e];
        dgm += g[e] * Sc[e];
      }
      j->dgamma[(b * T + t) * H + hh] = dgm;
      for (int64_t r = 0; r < R; ++r) {
        const double* xv = j->x + (((b * T + t) * R + r) * H + hh) * P;
        const double* bv = j->B + (((b * T + t) * R + r) * G + g_) * N;
        for (int64_t p = 0; p < P; ++p) {
          double s = 0.0;
          for (int64_t n = 0; n < N; ++n) s += dS[p * N + n] * bv[n];
          j->dx[(((b * T + t) * R + r) * H + hh) * P + p] = s;
        }
        for (int64_t n = 0; n < N; ++n) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p) s += dS[p * N + n] * xv[p];
          dBl[(t * R + r) * N + n] += s;
        }
      }
      if (j->theta && j->dtheta) {
        double* dth = j->dtheta + ((b * T + t) * H + hh) * (N / 2);
        for (int64_t k = 0; k < N / 2; ++k) {
          double s = 0.0;
          for (int64_t p = 0; p < P; ++p)
            s += g[p * N + 2 * k + 1] * v[p * N + 2 * k] - g[p * N + 2 * k] * v[p * N + 2 * k + 1];
          dth[k] = s;
        }
      }
      /* du = R(-theta_t) g, kept in g */
      if (j->theta) bwd_turn(j->theta + ((b * T + t) * H + hh) * (N / 2), P, N, -1.0, g);
      double da = 0.0, dbt = 0.0;
      for (int64_t e = 0; e < PN; ++e) {
        da += g[e] * hprev[e];
        dbt += g[e] * Sp[e];
      }
      j->ddA[(b * T + t) * H + hh] = a * da;
      j->dbeta[(b * T + t) * H + hh] = dbt;
      if (j->mutation == MUT_TBWD_NO_BETA_CARRY) {
        /* the planted mistake: the beta term's gradient is not carried to S_{t-1} */
        for (int64_t e = 0; e < PN; ++e) dS[e] = 0.0;
      } else {
        for (int64_t e = 0; e < PN; ++e) dS[e] = bt * g[e];
      }
      for (int64_t e = 0; e < PN; ++e) g[e] *= a;
    }
  }
  if (j->dinit) memcpy(j->dinit + ((b * H + hh) * P) * N, g, sizeof(double) * PN);
  /* dS now holds dL/dS_{-1} */
  memset(dpB, 0, sizeof(double) * R * N);
  if (j->prev_x) {
    for (int64_t r = 0; r < R; ++r) {
      const double* pbv = j->prev_B + ((b * R + r) * G + g_) * N;
      const double* pxv = j->prev_x + ((b * R + r) * H + hh) * P;
      for (int64_t p = 0; p < P; ++p) {
        double s = 0.0;
        for (int64_t n = 0; n < N; ++n) s += dS[p * N + n] * pbv[n];
        if (j->dprev_x) j->dprev_x[((b * R + r) * H + hh) * P + p] = s;
      }
      for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t p = 0; p < P; ++p) s += dS[p * N + n] * pxv[p];
        dpB[r * N + n] = s;
      }
    }
  }
  pthread_mutex_lock(j->lock);
  for (int64_t t = 0; t < T; ++t)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t n = 0; n < N; ++n) {
        const int64_t o = (((b * T + t) * R + r) * G + g_) * N + n;
        j->dB[o] += dBl[(t * R + r) * N + n];
        j->dC[o] += dCl[(t * R + r) * N + n];
      }
  if (j->prev_x && j->dprev_B)
    for (int64_t r = 0; r < R; ++r)
      for (int64_t n = 0; n < N; ++n) j->dprev_B[((b * R + r) * G + g_) * N + n] += dpB[r * N + n];
  pthread_mutex_unlock(j->lock);
}

static void* tbwd_worker(void* arg) {
  const tbwd_job* j = (const tbwd_job*)arg;
  const int64_t PN = j->P * j->N, nck = (j->T + ORACLE_CKPT - 1) / ORACLE_CKPT;
  double* ck = (double*)malloc(sizeof(double) * PN * (size_t)nck);
  double* seg = (double*)malloc(sizeof(double) * PN * (ORACLE_CKPT + 1));
  double* buf = (double*)malloc(sizeof(double) * PN * 7);
  double* dBl = (double*)malloc(sizeof(double) * j->T * j->R * j->N);
  double* dCl = (double*)malloc(sizeof(double) * j->T * j->R * j->N);
  double* dpB = (double*)malloc(sizeof(double) * j->R * j->N);
  void* rc = NULL;
  if (!ck || !seg || !buf || !dBl || !dCl || !dpB) {
    rc = (void*)1;
  } else {
    for (int64_t idx = j->tid; idx < j->batch * j->H; idx += j->nthreads)
      tbwd_one(j, idx / j->H, idx % j->H, ck, seg, buf, buf + PN, buf + 2 * PN, buf + 3 * PN,
               buf + 4 * PN, buf + 5 * PN, buf + 6 * PN, dBl, dCl, dpB);
  }
  free(ck);
  free(seg);
  free(buf);
  free(dBl);
  free(dCl);
  free(dpB);
  return rc;
}

/* Backward of the trapezoidal SSD (theta, init_state, prev_x/prev_B, dfinal nullable; prev_x and
 * prev_B both or neither).  dB, dC, dprev_B are zeroed here; dtheta (needs theta), dinit,
 * dprev_x, dprev_B (need prev_x) nullable.  Returns 0 or a negative error. */
int oracle_ssd_trap_backward_ex(const double* x, const double* dA, const double* B,
                                const double* C, const double* gamma, const double* beta,
                                const double* theta, const double* init_state,
                                const double* prev_x, const double* prev_B, const double* dy,
                                const double* dfinal, double* dx, double* ddA, double* dB,
                                double* dC, double* dgamma, double* dbeta, double* dtheta,
                                double* dinit, double* dprev_x, double* dprev_B, int64_t batch,
                                int64_t T, int64_t R, int64_t H, int64_t G, int64_t P, int64_t N,
                                int64_t nthreads, int mutation) {
  if (!x || !dA || !B || !C || !gamma || !beta || !dy || !dx || !ddA || !dB || !dC || !dgamma ||
      !dbeta)
    return -1;
  if (batch < 1 || T < 1 || R < 1 || H < 1 || G < 1 || P < 1 || N < 1) return -2;
  if (H % G != 0) return -3;
  if (theta && (N % 2) != 0) return -4;
  if ((prev_x == NULL) != (prev_B == NULL)) return -6;
  memset(dB, 0, sizeof(double) * (size_t)(batch * T * R * G * N));
  memset(dC, 0, sizeof(double) * (size_t)(batch * T * R * G * N));
  if (dprev_B) memset(dprev_B, 0, sizeof(double) * (size_t)(batch * R * G * N));
  if (dprev_x) memset(dprev_x, 0, sizeof(double) * (size_t)(batch * R * H * P));
  const int64_t nt = clamp_threads(nthreads, batch * H);
  tbwd_job* jobs = (tbwd_job*)calloc((size_t)nt, sizeof(tbwd_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  pthread_mutex_t lock;
  if (!jobs || !th || pthread_mutex_init(&lock, NULL) != 0) {
    free(jobs);
    free(th);
    return -5;
  }
  for (int64_t i = 0; i < nt; ++i) {
    tbwd_job jb = {x,      dA,     B,      C,     gamma, beta,  theta,   init_state, prev_x,
                   prev_B, dy,     dfinal, dx,    ddA,   dB,    dC,      dgamma,     dbeta,
                   dtheta, dinit,  dprev_x, dprev_B, batch, T,  R,       H,          G,
                   P,      N,      mutation, nt,  i,     &lock};
    jobs[i] = jb;
  }
  int rc = 0;
  for (int64_t i = 1; i < nt; ++i) pthread_create(&th[i], NULL, tbwd_worker, &jobs[i]);
  if (tbwd_worker(&jobs[0]) != NULL) rc = -5;
  for (int64_t i = 1; i < nt; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret != NULL) rc = -5;
  }
  pthread_mutex_destroy(&lock);
  free(jobs);
  free(th);
  return rc;
}

/* ---------------------------------------------------------------------------------------- */
/* Selective scan                                                                            */
/* ---------------------------------------------------------------------------------------- */

typedef struct {
  const double *u, *delta, *A, *B, *C, *skip;
  double* y;
  int64_t batch, T, D, N;
  int mutation;
  int64_t nthreads, tid;
} ss_job;

static void* ss_worker(void* arg) {
  const ss_job* j = (const ss_job*)arg;
  const int64_t T = j->T, D = j->D, N = j->N;
  double* h = (double*)malloc(sizeof(double) * N);
  if (!h) return (void*)1;
  for (int64_t idx = j->tid; idx < j->batch * D; idx += j->nthreads) {
    const int64_t b = idx / D, d = idx % D;
    for (int64_t n = 0; n < N; ++n) h[n] = 0.0;
    const double sk = (j->skip && j->mutation != MUT_SS_NO_SKIP) ? j->skip[d] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
      const double dt = j->delta[(b * T + t) * D + d];
      const double uv = j->u[(b * T + t) * D + d];
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        const double abar = exp(dt * j->A[d * N + n]);
        const double bbar =
            (j->mutation == MUT_SS_DELTA_B) ? j->B[(b * T + t) * N + n] : dt * j->B[(b * T + t) * N + n];
        h[n] = abar * h[n] + bbar * uv;
        acc += j->C[(b * T + t) * N + n] * h[n];
      }
      j->y[(b * T + t) * D + d] = acc + sk * uv;
    }
  }
  free(h);
  return NULL;
}

int oracle_selective_scan_ex(const double* u, const double* delta, const double* A,
                             const double* B, const double* C, const double* skip, double* y,
                             int64_t batch, int64_t T, int64_t D, int64_t N, int64_t nthreads,
                             int mutation) {
  if (!u || !delta || !A || !B || !C || !y) return -1;
  if (batch < 0 || T < 0 || D < 1 || N < 1) return -2;
  if (batch == 0 || T == 0) return 0;
  const int64_t nt = clamp_threads(nthreads, batch * D);
  ss_job* jobs = (ss_job*)calloc((size_t)nt, sizeof(ss_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return -5;
  }
  int rc = 0;
  for (int64_t i = 0; i < nt; ++i) {
    ss_job j = {u, delta, A, B, C, skip, y, batch, T, D, N, mutation, nt, i};
    jobs[i] = j;
  }
  for (int64_t i = 1; i < nt; ++i) pthread_create(&th[i], NULL, ss_worker, &jobs[i]);
  if (ss_worker(&jobs[0]) != NULL) rc = -5;
  for (int64_t i = 1; i < nt; ++i) {
    void* ret = NULL;
    pthread_join(th[i], &ret);
    if (ret != NULL) rc = -5;
  }
  free(jobs);
  free(th);
  return rc;
}

int oracle_selective_scan(const double* u, const double* delta, const double* A, const double* B,
                          const double* C, const double* skip, double* y, int64_t batch,
                          int64_t T, int64_t D, int64_t N, int64_t nthreads) {
  return oracle_selective_scan_ex(u, delta, A, B, C, skip, y, batch, T, D, N, nthreads, MUT_NONE);
}
