/*
 * forward_from_c.c -- calls libittt.so from plain C99 (no C++, no torch):
 * reads a layer's inputs from a binary file, copies them to the device with
 * the CUDA runtime, runs ittt_forward on a stream, checks ittt_stream_status
 * and writes O back to a file.
 *
 * Input file: int64 B, T, d, f, chunk; float eta (4 bytes); then H, X0
 * [B,T,d], W_gate, W_up [f,d], W_down0 [d,f], W_target [d,d] as bf16 (raw
 * 16-bit words) and conv_w [d,3] as fp32.  Output file: O [B,T,d] bf16.
 * Usage: forward_from_c <input> <output>; exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "ittt.h"

static ittt_tensor desc(void* data, int32_t dtype, int32_t ndim, const int64_t* shape) {
  ittt_tensor t;
  int64_t stride = 1;
  int k;
  t.data = data;
  t.dtype = dtype;
  t.ndim = ndim;
  for (k = 3; k >= 0; --k) {
    t.shape[k] = k < ndim ? shape[k] : 1;
    t.stride[k] = 0;
  }
  for (k = ndim - 1; k >= 0; --k) {
    t.stride[k] = stride;
    stride *= shape[k];
  }
  return t;
}

static void* upload(FILE* in, size_t bytes) {
  void* host = malloc(bytes);
  void* dev = NULL;
  if (host == NULL || fread(host, 1, bytes, in) != bytes) return NULL;
  if (cudaMalloc(&dev, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  free(host);
  return dev;
}

int main(int argc, char** argv) {
  int64_t hdr[5];
  float eta;
  FILE* in;
  FILE* out;
  void *H, *X0, *Wg, *Wu, *W0, *Wt, *cw, *O;
  void* host_o;
  size_t btd;
  cudaStream_t stream;
  ittt_status s;
  if (argc != 3) return 2;
  in = fopen(argv[1], "rb");
  if (in == NULL || fread(hdr, sizeof(int64_t), 5, in) != 5 || fread(&eta, 4, 1, in) != 1)
    return 3;
  {
    const int64_t B = hdr[0], T = hdr[1], d = hdr[2], f = hdr[3], chunk = hdr[4];
    const int64_t sh_btd[3] = {B, T, d}, sh_fd[2] = {f, d}, sh_df[2] = {d, f},
                  sh_dd[2] = {d, d}, sh_d3[2] = {d, 3};
    ittt_tensor tH, tX0, tWg, tWu, tW0, tWt, tcw, tO;
    btd = (size_t)(B * T * d);
    H = upload(in, btd * 2);
    X0 = upload(in, btd * 2);
    Wg = upload(in, (size_t)(f * d) * 2);
    Wu = upload(in, (size_t)(f * d) * 2);
    W0 = upload(in, (size_t)(d * f) * 2);
    Wt = upload(in, (size_t)(d * d) * 2);
    cw = upload(in, (size_t)(d * 3) * 4);
    fclose(in);
    if (!H || !X0 || !Wg || !Wu || !W0 || !Wt || !cw) return 4;
    if (cudaMalloc(&O, btd * 2) != cudaSuccess) return 5;
    tH = desc(H, ITTT_BF16, 3, sh_btd);
    tX0 = desc(X0, ITTT_BF16, 3, sh_btd);
    tWg = desc(Wg, ITTT_BF16, 2, sh_fd);
    tWu = desc(Wu, ITTT_BF16, 2, sh_fd);
    tW0 = desc(W0, ITTT_BF16, 2, sh_df);
    tWt = desc(Wt, ITTT_BF16, 2, sh_dd);
    tcw = desc(cw, ITTT_FP32, 2, sh_d3);
    tO = desc(O, ITTT_BF16, 3, sh_btd);
    if (cudaStreamCreate(&stream) != cudaSuccess) return 6;
    s = ittt_forward(&tH, &tX0, &tWg, &tWu, &tW0, &tWt, &tcw, eta, chunk, &tO,
                     (ittt_stream_t)stream);
    if (s == ITTT_OK) s = ittt_stream_status((ittt_stream_t)stream);
    if (s != ITTT_OK) {
      fprintf(stderr, "ittt: status %d: %s\n", (int)s, ittt_last_error());
      return 7;
    }
  }
  host_o = malloc(btd * 2);
  if (host_o == NULL || cudaMemcpy(host_o, O, btd * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 8;
  out = fopen(argv[2], "wb");
  if (out == NULL || fwrite(host_o, 1, btd * 2, out) != btd * 2) return 9;
  fclose(out);
  printf("forward_from_c: ok\n");
  return 0;
}
