/* The C ABI used from plain C, with no Python or torch: P device buffers from
 * cudaMalloc, a 4 x 2 torus plan, one all-reduce on the default stream, and a
 * check against the exact integer sums (integer-valued binary32 inputs whose
 * sums are exact in binary32, so every add order gives the same bits).
 * Prints "ok" and exits 0 on success. */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include "ddl.h"

#define P 8
#define N 100003

static int check(ddl_status_t s, const char* what) {
  if (s != DDL_OK) {
    fprintf(stderr, "%s: %s\n", what, ddl_status_string(s));
    return 1;
  }
  return 0;
}

int main(void) {
  float* host = (float*)malloc(sizeof(float) * (size_t)N * P);
  float* out = (float*)malloc(sizeof(float) * (size_t)N);
  long long* want = (long long*)calloc(N, sizeof(long long));
  void* bufs[P];
  if (!host || !out || !want) return 2;
  for (int r = 0; r < P; ++r)
    for (long i = 0; i < N; ++i) {
      const long v = (long)((r * 7919L + i * 104729L) % 2001L) - 1000L;
      host[(size_t)r * N + i] = (float)v;
      want[i] += v;
    }
  for (int r = 0; r < P; ++r) {
    if (cudaMalloc(&bufs[r], sizeof(float) * N) != cudaSuccess) return 3;
    if (cudaMemcpy(bufs[r], host + (size_t)r * N, sizeof(float) * N, cudaMemcpyHostToDevice) != cudaSuccess) return 3;
  }
  ddl_topology_t topo = {DDL_TORUS, 1, 4, 2};
  ddl_plan_t plan = NULL;
  if (check(ddl_plan_create(P, N, DDL_FP32, topo, 0, &plan), "ddl_plan_create")) return 4;
  if (check(ddl_allreduce(plan, bufs, 1.0f, NULL), "ddl_allreduce")) return 4;
  if (cudaDeviceSynchronize() != cudaSuccess) return 5;
  if (check(ddl_plan_check(plan), "ddl_plan_check")) return 4;
  int bad = 0;
  for (int r = 0; r < P && !bad; ++r) {
    if (cudaMemcpy(out, bufs[r], sizeof(float) * N, cudaMemcpyDeviceToHost) != cudaSuccess) return 5;
    for (long i = 0; i < N; ++i)
      if (out[i] != (float)want[i]) {
        fprintf(stderr, "rank %d element %ld: got %.1f want %lld\n", r, i, out[i], want[i]);
        bad = 1;
        break;
      }
  }
  ddl_plan_destroy(plan);
  for (int r = 0; r < P; ++r) cudaFree(bufs[r]);
  free(host);
  free(out);
  free(want);
  if (bad) return 6;
  printf("ok\n");
  return 0;
}
