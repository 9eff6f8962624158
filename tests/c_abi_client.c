/* A plain C client of libpdecode: the C ABI with no Python on the call path.
 *
 * Usage: c_abi_client DIR
 * DIR holds params.txt ("B Hq Hkv D block_size num_blocks max_blocks qlen
 * kv_dtype window num_splits scale k_scale v_scale") and the raw
 * little-endian arrays q.bin, k.bin, v.bin (element bytes as the kind says),
 * block_table.bin and seq_lens.bin (int32). The client copies them to device
 * memory it allocates with the CUDA runtime, sizes the workspace with
 * pd_workspace_bytes, runs decode_paged on a stream of its own and writes
 * out.bin (q's element type) and flag.txt (the device error bits).
 * Exit status: 0 on success, 1 on a file or CUDA error, 2 on a pd_status
 * other than PD_OK. Test infrastructure. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "pdecode.h"

static void* read_all(const char* dir, const char* name, size_t* bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  fseek(f, 0, SEEK_END);
  long n = ftell(f);
  fseek(f, 0, SEEK_SET);
  void* buf = malloc(n > 0 ? (size_t)n : 1);
  if (buf && n > 0 && fread(buf, 1, (size_t)n, f) != (size_t)n) {
    free(buf);
    buf = NULL;
  }
  fclose(f);
  *bytes = (size_t)n;
  return buf;
}

static void* to_device(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes > 0 ? bytes : 16) != cudaSuccess) return NULL;
  if (bytes > 0 && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(d);
    return NULL;
  }
  return d;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s DIR\n", argv[0]);
    return 1;
  }
  const char* dir = argv[1];
  char path[4096];
  snprintf(path, sizeof path, "%s/params.txt", dir);
  FILE* pf = fopen(path, "r");
  if (!pf) return 1;
  pd_dims d;
  int qlen, window, splits;
  float scale;
  int n = fscanf(pf, "%d %d %d %d %d %d %d %d %d %d %d %f %f %f", &d.B, &d.Hq, &d.Hkv, &d.D,
                 &d.block_size, &d.num_blocks, &d.max_blocks_per_seq, &qlen, &d.kv_dtype, &window,
                 &splits, &scale, &d.k_scale, &d.v_scale);
  fclose(pf);
  if (n != 14) return 1;

  const char* names[5] = {"q.bin", "k.bin", "v.bin", "block_table.bin", "seq_lens.bin"};
  void* host[5];
  void* dev[5];
  size_t bytes[5];
  for (int i = 0; i < 5; ++i) {
    host[i] = read_all(dir, names[i], &bytes[i]);
    if (!host[i]) return 1;
    dev[i] = to_device(host[i], bytes[i]);
    if (!dev[i]) return 1;
  }
  const size_t out_bytes = bytes[0];  /* out has q's shape and type */
  void* out = NULL;
  uint32_t* flag = NULL;
  if (cudaMalloc(&out, out_bytes) != cudaSuccess || cudaMalloc((void**)&flag, 4) != cudaSuccess ||
      cudaMemset(flag, 0, 4) != cudaSuccess)
    return 1;
  const size_t ws_bytes = pd_workspace_bytes(&d, qlen, splits, 0);
  void* ws = NULL;
  if (ws_bytes > 0 && cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 1;
  cudaStream_t stream;
  if (cudaStreamCreate(&stream) != cudaSuccess) return 1;

  pd_status rc = decode_paged(dev[0], dev[1], dev[2], (const int32_t*)dev[3], (const int32_t*)dev[4], scale,
                              window, qlen, splits, out, &d, ws, ws_bytes, flag, stream);
  if (rc != PD_OK) {
    fprintf(stderr, "decode_paged: %s\n", pd_status_str(rc));
    return 2;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) return 1;

  void* out_host = malloc(out_bytes);
  uint32_t flag_host = 0;
  if (!out_host || cudaMemcpy(out_host, out, out_bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(&flag_host, flag, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 1;
  snprintf(path, sizeof path, "%s/out.bin", dir);
  FILE* of = fopen(path, "wb");
  if (!of || fwrite(out_host, 1, out_bytes, of) != out_bytes) return 1;
  fclose(of);
  snprintf(path, sizeof path, "%s/flag.txt", dir);
  FILE* ff = fopen(path, "w");
  if (!ff) return 1;
  fprintf(ff, "%u\n", flag_host);
  fclose(ff);

  cudaStreamDestroy(stream);
  for (int i = 0; i < 5; ++i) {
    cudaFree(dev[i]);
    free(host[i]);
  }
  cudaFree(out);
  cudaFree(flag);
  if (ws) cudaFree(ws);
  free(out_host);
  return 0;
}
