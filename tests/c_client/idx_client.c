/*
 * A plain C client of include/idx.h: no Python, no torch.  It reads one indexer
 * problem from raw little-endian files in a directory, runs idx_launch_host on
 * host buffers (pageable memory, so the copies are synchronous), and writes the
 * [R][K] int32 result to out.bin in the same directory.  It also checks that bad
 * arguments come back as IDX_EINVAL before anything is launched.
 *
 * Files: meta.txt holds "R Q P pt_stride max_bound kv_dtype K rows_hint";
 * q.bin (bf16 [R][64][128]), w.bin (fp32 [R][64]), k_cache.bin, k_scale.bin
 * (fp32 [P][64], E4M3 only), page_table.bin (int32 [Q][pt_stride]), row_req.bin
 * and row_bound.bin (int32 [R]).
 *
 * Exit status 0 on success; a message on stderr and a non-zero status otherwise.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "idx.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (f == NULL) {
    fprintf(stderr, "cannot open %s\n", path);
    exit(2);
  }
  void *p = malloc(bytes > 0 ? bytes : 1);
  if (p == NULL || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read of %s (%zu bytes expected)\n", path, bytes);
    exit(2);
  }
  fclose(f);
  return p;
}

int main(int argc, char **argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s <problem directory>\n", argv[0]);
    return 2;
  }
  const char *dir = argv[1];
  char meta_path[4096];
  snprintf(meta_path, sizeof meta_path, "%s/meta.txt", dir);
  FILE *mf = fopen(meta_path, "r");
  long long R, Q, P, stride, max_bound, kv, K, hint;
  if (mf == NULL || fscanf(mf, "%lld %lld %lld %lld %lld %lld %lld %lld", &R, &Q, &P, &stride, &max_bound, &kv, &K,
                           &hint) != 8) {
    fprintf(stderr, "cannot read %s\n", meta_path);
    return 2;
  }
  fclose(mf);
  const size_t key_bytes = (size_t)P * IDX_PAGE * IDX_DIM * (kv == IDX_KV_E4M3 ? 1 : 2);

  idx_problem p;
  memset(&p, 0, sizeof p);
  p.q = read_file(dir, "q.bin", (size_t)R * IDX_HEADS * IDX_DIM * 2);
  p.w = (const float *)read_file(dir, "w.bin", (size_t)R * IDX_HEADS * 4);
  p.k_cache = read_file(dir, "k_cache.bin", key_bytes);
  p.k_scale = kv == IDX_KV_E4M3 ? (const float *)read_file(dir, "k_scale.bin", (size_t)P * IDX_PAGE * 4) : NULL;
  p.page_table = (const int32_t *)read_file(dir, "page_table.bin", (size_t)Q * stride * 4);
  p.row_req = (const int32_t *)read_file(dir, "row_req.bin", (size_t)R * 4);
  p.row_bound = (const int32_t *)read_file(dir, "row_bound.bin", (size_t)R * 4);
  p.R = (int32_t)R;
  p.Q = (int32_t)Q;
  p.P = P;
  p.pt_stride = (int32_t)stride;
  p.max_bound = (int32_t)max_bound;
  p.kv_dtype = (int32_t)kv;
  p.rows_hint = (int32_t)hint;

  /* argument checks that must refuse before launching anything */
  int32_t *host_out = (int32_t *)malloc((size_t)R * K * 4);
  if (idx_launch_host(&p, (int32_t)K, NULL, NULL, 0, NULL) != IDX_EINVAL ||
      idx_launch_host(&p, IDX_MAX_K + 1, host_out, NULL, 0, NULL) != IDX_EINVAL ||
      idx_workspace_size(NULL, (int32_t)K) != 0) {
    fprintf(stderr, "bad arguments were not refused\n");
    return 1;
  }

  const size_t arena_bytes = idx_host_arena_size(&p, (int32_t)K);
  if (arena_bytes == 0) {
    fprintf(stderr, "idx_host_arena_size refused the problem\n");
    return 1;
  }
  void *arena = NULL;
  if (cudaMalloc(&arena, arena_bytes) != cudaSuccess) {
    fprintf(stderr, "cudaMalloc of %zu bytes failed\n", arena_bytes);
    return 1;
  }
  const idx_status st = idx_launch_host(&p, (int32_t)K, host_out, arena, arena_bytes, NULL);
  if (st != IDX_OK) {
    fprintf(stderr, "idx_launch_host: %s\n", idx_status_string(st));
    return 1;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    fprintf(stderr, "CUDA error after the launch\n");
    return 1;
  }
  char out_path[4096];
  snprintf(out_path, sizeof out_path, "%s/out.bin", dir);
  FILE *of = fopen(out_path, "wb");
  if (of == NULL || fwrite(host_out, 4, (size_t)R * K, of) != (size_t)R * K) {
    fprintf(stderr, "cannot write %s\n", out_path);
    return 1;
  }
  fclose(of);
  cudaFree(arena);
  printf("idx_client: %s, version %d, R %lld, K %lld\n", idx_status_string(st), idx_version(), R, K);
  return 0;
}
