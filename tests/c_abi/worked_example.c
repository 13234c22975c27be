/* A plain C consumer of libccl: the worked example of "Networks and Collective
 * Communication" (section 4.1) through the C ABI alone -- no Python, no torch.
 *
 * Usage: worked_example x0_0 .. x0_3 x1_0 .. x3_3   (the 4 x 4 fp32 inputs)
 * Prints one line per result in the layout of tests/golden/worked_example_p4.txt
 * ("name: v v v v"); the test compares them with that file.  Exit status 0
 * when every call returned CCL_OK, 1 otherwise (the failing call is named on
 * stderr). */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "ccl.h"

enum { P = 4, N = 4 };

static int check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
  }
  return 0;
}

static int check_ccl(ccl_status_t st, const char* what) {
  if (st != CCL_OK) {
    fprintf(stderr, "%s: %s (%s)\n", what, ccl_status_string(st), ccl_last_error());
    return 1;
  }
  return 0;
}

/* copy `count` floats back from the device and print them after `name` */
static int print_dev(const char* name, const float* dev, int count) {
  float h[P * N];
  if (check_cuda(cudaMemcpy(h, dev, sizeof(float) * (size_t)count, cudaMemcpyDeviceToHost), name)) return 1;
  printf("%s:", name);
  for (int i = 0; i < count; ++i) printf(" %g", (double)h[i]);
  printf("\n");
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 1 + P * N) {
    fprintf(stderr, "usage: %s <16 fp32 inputs, rank-major>\n", argv[0]);
    return 2;
  }
  float host[P * N];
  for (int i = 0; i < P * N; ++i) host[i] = strtof(argv[1 + i], NULL);

  /* one device allocation: inputs, then the outputs of each call */
  float* base = NULL;
  if (check_cuda(cudaMalloc((void**)&base, sizeof(float) * 8 * P * N), "cudaMalloc")) return 1;
  float* in = base;                /* P x N inputs */
  float* ar = base + 1 * P * N;    /* all-reduce outputs */
  float* rs = base + 2 * P * N;    /* reduce-scatter shards (len(k) = 1) */
  float* ag = base + 3 * P * N;    /* all-gather outputs */
  float* a2a = base + 4 * P * N;   /* all-to-all outputs */
  float* bc = base + 5 * P * N;    /* broadcast outputs */
  float* red = base + 6 * P * N;   /* reduce output on the root */
  if (check_cuda(cudaMemcpy(in, host, sizeof host, cudaMemcpyHostToDevice), "copy in")) return 1;

  const void* send[P];
  void* recv_ar[P];
  void* recv_rs[P];
  const void* ag_send[P];
  void* recv_ag[P];
  void* recv_a2a[P];
  void* recv_bc[P];
  for (int r = 0; r < P; ++r) {
    send[r] = in + r * N;
    recv_ar[r] = ar + r * N;
    recv_rs[r] = rs + r;
    ag_send[r] = in + r * N + r; /* device d contributes block d of its own vector */
    recv_ag[r] = ag + r * N;
    recv_a2a[r] = a2a + r * N;
    recv_bc[r] = bc + r * N;
  }
  int bad = 0;
  bad |= check_ccl(ccl_allreduce(send, recv_ar, P, N, CCL_F32, CCL_SUM, NULL), "ccl_allreduce");
  bad |= check_ccl(ccl_reduce_scatter(send, recv_rs, P, N, CCL_F32, CCL_SUM, NULL), "ccl_reduce_scatter");
  bad |= check_ccl(ccl_all_gather(ag_send, recv_ag, P, N, CCL_F32, NULL), "ccl_all_gather");
  bad |= check_ccl(ccl_all_to_all(send, recv_a2a, P, N, CCL_F32, NULL), "ccl_all_to_all");
  bad |= check_ccl(ccl_broadcast(in, recv_bc, P, N, CCL_F32, 0, NULL), "ccl_broadcast");
  bad |= check_ccl(ccl_reduce(send, red, P, N, CCL_F32, CCL_SUM, 0, NULL), "ccl_reduce");
  bad |= check_ccl(ccl_stream_check(NULL), "ccl_stream_check");
  if (bad) return 1;

  char name[32];
  bad |= print_dev("allreduce", ar, N);
  for (int k = 0; k < P; ++k) {
    snprintf(name, sizeof name, "reduce_scatter %d", k);
    bad |= print_dev(name, rs + k, 1);
  }
  bad |= print_dev("all_gather", ag, N);
  for (int j = 0; j < P; ++j) {
    snprintf(name, sizeof name, "all_to_all %d", j);
    bad |= print_dev(name, a2a + j * N, N);
  }
  bad |= print_dev("broadcast_root0", bc + 3 * N, N);
  bad |= print_dev("reduce_root0", red, N);

  /* every rank of the all-reduce and the all-gather holds the same values */
  float h[8 * P * N];
  bad |= check_cuda(cudaMemcpy(h, base, sizeof h, cudaMemcpyDeviceToHost), "copy out");
  for (int r = 1; r < P && !bad; ++r)
    for (int i = 0; i < N; ++i)
      if (h[P * N + r * N + i] != h[P * N + i] || h[3 * P * N + r * N + i] != h[3 * P * N + i]) {
        fprintf(stderr, "rank %d differs from rank 0\n", r);
        bad = 1;
      }
  cudaFree(base);
  return bad ? 1 : 0;
}
