/* A whole update driven through the C ABI from plain C: plan, reduce (two
 * microbatches), norm, clip + AdamW; the update writing per-tensor buffers;
 * the update of every rank's shard view; device memory from the CUDA
 * runtime, no other framework.  Checked against the CPU oracle (linked
 * separately; test infrastructure) at the suite's tolerances.  Exit 0 on
 * success, 1 on a mismatch, 2 on an API error. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "grs.h"

/* the oracle's entry points used here (its own header is not included: the
 * library and the oracle share nothing) */
int oracle_plan(const int64_t*, const int32_t*, int32_t, int32_t, int32_t, int32_t, int32_t, int64_t, int32_t,
                int32_t*, int32_t*, int64_t*, int32_t*, int64_t*, int64_t*, int64_t*, int64_t*);
int oracle_reduce_bucket(int32_t, int32_t, int32_t, int32_t, int64_t, int64_t, int32_t, const uint16_t*, double*);
double oracle_norm_sq(const double*, int64_t, int32_t);
double oracle_clip_coef(double, double);
void oracle_adamw(int64_t, int64_t, const double*, int32_t, double, const double*, int32_t, const float*,
                  const float*, const float*, float*, float*, float*, uint16_t*);

#define CHECK(x) do { grs_status s_ = (x); if (s_ != GRS_OK) { fprintf(stderr, "%s: %d %s\n", #x, (int)s_, grs_last_error()); return 2; } } while (0)
#define CUDA(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)

static uint32_t lcg = 12345u;
static float frand(void) { /* uniform in [-1, 1) */
  lcg = lcg * 1664525u + 1013904223u;
  return (float)((lcg >> 8) & 0xFFFFFF) / 8388608.0f - 1.0f;
}
static uint16_t to_bf16(float x) { /* truncation is enough for test data */
  uint32_t w;
  memcpy(&w, &x, 4);
  return (uint16_t)(w >> 16);
}
static int close_enough(double got, double want) { return fabs(got - want) <= 1e-7 + 1e-5 * fabs(want); }

int main(void) {
  const int64_t numels[] = {3001, 77, 2048, 9, 500};
  const int32_t owners[] = {GRS_REPLICA_AVG, GRS_PARTIAL_SUM, GRS_LOCAL_SHARD, GRS_ALREADY_REDUCED,
                            GRS_REPLICA_AVG};
  const int32_t n = 5, world = 8, tp = 2, dr = 2, ds = 2, M = 2;
  const int64_t bucket_bytes = 4096;
  grs_plan* plan = NULL;
  CHECK(grs_plan_create(numels, owners, n, world, tp, dr, ds, bucket_bytes, 0, &plan));
  grs_plan_info info;
  CHECK(grs_plan_query(plan, &info));
  const int64_t nrp = info.n_rank_pad, nsp = info.n_state_pad;

  /* host inputs: M microbatches x world ranks, bf16 */
  uint16_t* host = (uint16_t*)malloc(sizeof(uint16_t) * M * world * nrp);
  for (int64_t i = 0; i < M * world * nrp; ++i) host[i] = to_bf16(1e-3f * frand());
  float* master0 = (float*)malloc(sizeof(float) * nsp);
  for (int64_t i = 0; i < nsp; ++i) master0[i] = 0.02f * frand();

  void* d_grads[2][8];
  for (int j = 0; j < M; ++j)
    for (int k = 0; k < world; ++k) {
      CUDA(cudaMalloc(&d_grads[j][k], sizeof(uint16_t) * nrp));
      CUDA(cudaMemcpy(d_grads[j][k], host + ((int64_t)j * world + k) * nrp, sizeof(uint16_t) * nrp,
                      cudaMemcpyHostToDevice));
    }
  float *acc, *master, *m, *v;
  uint16_t* params;
  double* norm;
  void* ws;
  CUDA(cudaMalloc((void**)&acc, sizeof(float) * nsp));
  CUDA(cudaMalloc((void**)&master, sizeof(float) * nsp));
  CUDA(cudaMalloc((void**)&m, sizeof(float) * nsp));
  CUDA(cudaMalloc((void**)&v, sizeof(float) * nsp));
  CUDA(cudaMalloc((void**)&params, sizeof(uint16_t) * nsp));
  CUDA(cudaMalloc((void**)&norm, sizeof(double)));
  CUDA(cudaMalloc(&ws, (size_t)info.workspace_bytes));
  CUDA(cudaMemset(ws, 0, (size_t)info.workspace_bytes));
  CUDA(cudaMemcpy(master, master0, sizeof(float) * nsp, cudaMemcpyHostToDevice));
  CUDA(cudaMemset(m, 0, sizeof(float) * nsp));
  CUDA(cudaMemset(v, 0, sizeof(float) * nsp));

  cudaStream_t st;
  CUDA(cudaStreamCreate(&st));
  for (int j = 0; j < M; ++j)
    CHECK(grs_reduce_all(plan, (const void* const*)d_grads[j], acc, j > 0, j == M - 1, ws, st));
  CHECK(grs_grad_norm_sq(plan, acc, M, ws, 1, norm, st));
  grs_adamw hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 1.0f, 1, M};
  CHECK(grs_clip_adamw_step(plan, &hp, norm, acc, master, m, v, params, st));
  CHECK(grs_check_device_errors(plan, st));

  float* h_acc = (float*)malloc(sizeof(float) * nsp);
  float* h_master = (float*)malloc(sizeof(float) * nsp);
  double h_norm = 0.0;
  CUDA(cudaMemcpy(h_acc, acc, sizeof(float) * nsp, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(h_master, master, sizeof(float) * nsp, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(&h_norm, norm, sizeof(double), cudaMemcpyDeviceToHost));

  /* oracle: its own plan, the same bytes */
  int32_t dims[4], t_bucket[5], b_tag[5];
  int64_t t_off[5], b_pad[5], b_used[5], b_roff[5], b_soff[5];
  if (oracle_plan(numels, owners, n, world, tp, dr, ds, bucket_bytes, 5, dims, t_bucket, t_off, b_tag, b_pad,
                  b_used, b_roff, b_soff) != 0) return 2;
  const int nb = dims[3];
  if (nb != info.n_buckets) { fprintf(stderr, "bucket count differs\n"); return 1; }
  double* oacc = (double*)calloc((size_t)nsp, sizeof(double));
  for (int b = 0; b < nb; ++b) {
    const int64_t P = b_pad[b];
    uint16_t* g = (uint16_t*)malloc(sizeof(uint16_t) * M * world * (P ? P : 1));
    for (int j = 0; j < M; ++j)
      for (int k = 0; k < world; ++k)
        memcpy(g + ((int64_t)j * world + k) * P, host + ((int64_t)j * world + k) * nrp + b_roff[b],
               sizeof(uint16_t) * P);
    if (oracle_reduce_bucket(b_tag[b], tp, dr, ds, P, b_used[b], M, g, oacc + b_soff[b]) != 0) return 2;
    free(g);
  }
  const double s = oracle_norm_sq(oacc, nsp, M);
  const double c = oracle_clip_coef(s, 1.0);
  float* om = (float*)calloc((size_t)nsp, sizeof(float));
  float* ov = (float*)calloc((size_t)nsp, sizeof(float));
  float* op = (float*)calloc((size_t)nsp, sizeof(float));
  float* z = (float*)calloc((size_t)nsp, sizeof(float));
  uint16_t* ob = (uint16_t*)calloc((size_t)nsp, sizeof(uint16_t));
  const double hpd[5] = {hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay};
  for (int b = 0; b < nb; ++b) {
    const int copies = b_tag[b] == GRS_LOCAL_SHARD ? tp : 1;
    for (int t = 0; t < copies; ++t) {
      const int64_t o = b_soff[b] + (int64_t)t * b_pad[b];
      oracle_adamw(b_pad[b], b_used[b], oacc + o, M, c, hpd, 1, master0 + o, z + o, z + o, op + o, om + o, ov + o,
                   ob + o);
    }
  }
  int bad = 0;
  if (!close_enough(h_norm, s)) { fprintf(stderr, "norm %g vs %g\n", h_norm, s); bad = 1; }
  for (int64_t i = 0; i < nsp && bad < 5; ++i) {
    if (!close_enough(h_acc[i], oacc[i])) { fprintf(stderr, "acc[%lld] %g vs %g\n", (long long)i, h_acc[i], oacc[i]); ++bad; }
    if (!close_enough(h_master[i], op[i])) { fprintf(stderr, "master[%lld] %g vs %g\n", (long long)i, h_master[i], op[i]); ++bad; }
  }
  printf("c-abi update: %d buckets, %lld state elements, norm^2 %.9g (oracle %.9g): %s\n", nb, (long long)nsp, h_norm,
         s, bad ? "MISMATCH" : "ok");

  /* The same update again from the initial state, with the bf16 parameters
   * written straight into per-tensor buffers (no bucket-ordered copy): each
   * tensor must hold, bit for bit, the bf16 values the first update wrote at
   * its segments (tp rows concatenated for LOCAL_SHARD). */
  uint16_t* h_params = (uint16_t*)malloc(sizeof(uint16_t) * nsp);
  CUDA(cudaMemcpy(h_params, params, sizeof(uint16_t) * nsp, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(master, master0, sizeof(float) * nsp, cudaMemcpyHostToDevice));
  CUDA(cudaMemset(m, 0, sizeof(float) * nsp));
  CUDA(cudaMemset(v, 0, sizeof(float) * nsp));
  uint16_t* d_tensor[5];
  for (int i = 0; i < n; ++i) CUDA(cudaMalloc((void**)&d_tensor[i], sizeof(uint16_t) * numels[i]));
  uint16_t** d_table;
  CUDA(cudaMalloc((void**)&d_table, sizeof(uint16_t*) * n));
  CUDA(cudaMemcpy(d_table, d_tensor, sizeof(uint16_t*) * n, cudaMemcpyHostToDevice));
  CHECK(grs_clip_adamw_step_to_tensors(plan, &hp, norm, acc, master, m, v, NULL, (uint16_t* const*)d_table, st));
  CHECK(grs_check_device_errors(plan, st));
  int bad_t = 0;
  for (int b = 0; b < nb; ++b) {
    grs_bucket_desc bd;
    CHECK(grs_bucket_info(plan, b, &bd));
    for (int i = 0; i < bd.n_segments; ++i) {
      grs_segment_desc sd;
      CHECK(grs_segment_info(plan, b, i, &sd));
      uint16_t* got = (uint16_t*)malloc(sizeof(uint16_t) * (sd.numel ? sd.numel : 1));
      CUDA(cudaMemcpy(got, d_tensor[sd.tensor] + sd.tensor_offset, sizeof(uint16_t) * sd.numel,
                      cudaMemcpyDeviceToHost));
      if (memcmp(got, h_params + sd.state_offset, sizeof(uint16_t) * sd.numel) != 0) ++bad_t;
      free(got);
    }
  }
  printf("c-abi update to tensors: %s\n", bad_t ? "MISMATCH" : "ok");

  /* Shard views: every rank (s, t) of one replica, given its slices of the
   * reduced gradient and of the initial state, updates its shard exactly as
   * the plan's own update did (same S). */
  float* h_master2 = (float*)malloc(sizeof(float) * nsp);
  CUDA(cudaMemcpy(h_master2, master, sizeof(float) * nsp, cudaMemcpyDeviceToHost));
  int bad_v = 0;
  for (int t = 0; t < tp; ++t)
    for (int sh = 0; sh < ds; ++sh) {
      grs_plan* view = NULL;
      CHECK(grs_plan_shard_view(plan, sh, t, &view));
      grs_plan_info vi;
      CHECK(grs_plan_query(view, &vi));
      const int64_t nv = vi.n_state_pad > 0 ? vi.n_state_pad : 1;
      float* h_acc_v = (float*)malloc(sizeof(float) * nv);
      float* h_m0_v = (float*)malloc(sizeof(float) * nv);
      float* want_v = (float*)malloc(sizeof(float) * nv);
      for (int b = 0; b < nb; ++b) {
        grs_bucket_desc pb, vb;
        CHECK(grs_bucket_info(plan, b, &pb));
        CHECK(grs_bucket_info(view, b, &vb));
        const int row = pb.tag == GRS_LOCAL_SHARD ? t : 0;
        const int64_t src = pb.state_offset + (int64_t)row * pb.padded + (int64_t)sh * pb.shard_len;
        memcpy(h_acc_v + vb.state_offset, h_acc + src, sizeof(float) * vb.padded);
        memcpy(h_m0_v + vb.state_offset, master0 + src, sizeof(float) * vb.padded);
        memcpy(want_v + vb.state_offset, h_master2 + src, sizeof(float) * vb.padded);
      }
      float *acc_v, *master_v, *m_v, *v_v;
      uint16_t* params_v;
      CUDA(cudaMalloc((void**)&acc_v, sizeof(float) * nv));
      CUDA(cudaMalloc((void**)&master_v, sizeof(float) * nv));
      CUDA(cudaMalloc((void**)&m_v, sizeof(float) * nv));
      CUDA(cudaMalloc((void**)&v_v, sizeof(float) * nv));
      CUDA(cudaMalloc((void**)&params_v, sizeof(uint16_t) * nv));
      CUDA(cudaMemcpy(acc_v, h_acc_v, sizeof(float) * vi.n_state_pad, cudaMemcpyHostToDevice));
      CUDA(cudaMemcpy(master_v, h_m0_v, sizeof(float) * vi.n_state_pad, cudaMemcpyHostToDevice));
      CUDA(cudaMemset(m_v, 0, sizeof(float) * nv));
      CUDA(cudaMemset(v_v, 0, sizeof(float) * nv));
      CHECK(grs_clip_adamw_step(view, &hp, norm, acc_v, master_v, m_v, v_v, params_v, st));
      CHECK(grs_check_device_errors(view, st));
      float* got_v = (float*)malloc(sizeof(float) * nv);
      CUDA(cudaMemcpy(got_v, master_v, sizeof(float) * vi.n_state_pad, cudaMemcpyDeviceToHost));
      if (memcmp(got_v, want_v, sizeof(float) * vi.n_state_pad) != 0) ++bad_v;
      cudaFree(acc_v); cudaFree(master_v); cudaFree(m_v); cudaFree(v_v); cudaFree(params_v);
      free(h_acc_v); free(h_m0_v); free(want_v); free(got_v);
      grs_plan_destroy(view);
    }
  printf("c-abi shard views: %s\n", bad_v ? "MISMATCH" : "ok");
  grs_plan_destroy(plan);
  return (bad || bad_t || bad_v) ? 1 : 0;
}
