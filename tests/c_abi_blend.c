/* A blended prefill driven from C through include/cacheblend.h alone: the
 * CUDA runtime for memory, the library for every step.  It reads a model,
 * its chunks and a query from the input file, prefills each chunk on its own
 * (cb_full_prefill), blends the request (cb_blend_prefill, token top-k) and
 * writes the selection, the computed rows, their hidden states and the first
 * token to the output file.
 *
 * Input (little-endian): int32 n_layers, d_model, n_q_heads, n_kv_heads,
 * head_dim, d_ffn, vocab, max_positions, n_chunks, n_query, ratio_bp;
 * float32 rope_base, norm_eps; int32 chunk_len[n_chunks]; float32 embed
 * [vocab][d], final_norm [d], then per layer w_qkv, w_o, w_gate, w_up,
 * w_down, norm1, norm2; int32 tokens [sum chunk_len + n_query].
 * Output: int32 K, R, first_token; int32 selected[K]; int32 rows[R];
 * float32 hidden[R][d].  Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "cacheblend.h"

static FILE *in;

static void die(const char *what) {
  fprintf(stderr, "c_abi_blend: %s\n", what);
  exit(1);
}
static void need(cb_status s, const char *what) {
  if (s != CB_OK) {
    fprintf(stderr, "c_abi_blend: %s: status %d: %s\n", what, (int)s, cb_last_error_message());
    exit(1);
  }
}
static void cuda(cudaError_t e, const char *what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "c_abi_blend: %s: %s\n", what, cudaGetErrorString(e));
    exit(1);
  }
}
static void read_all(void *dst, size_t bytes) {
  if (fread(dst, 1, bytes, in) != bytes) die("short input file");
}
static void *dev_alloc(size_t bytes) {
  void *p = NULL;
  cuda(cudaMalloc(&p, bytes ? bytes : 16), "cudaMalloc");
  return p;
}
/* a host array of `count` elements of `size` bytes from the input, on the device */
static void *upload(size_t count, size_t size) {
  const size_t bytes = count * size;
  void *h = malloc(bytes > 0 ? bytes : 1);
  if (!h) die("out of host memory");
  read_all(h, bytes);
  void *d = dev_alloc(bytes);
  cuda(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice), "upload");
  free(h);
  return d;
}

int main(int argc, char **argv) {
  if (argc != 3) die("usage: c_abi_blend <input> <output>");
  in = fopen(argv[1], "rb");
  if (!in) die("cannot open the input file");
  int32_t hdr[11];
  float fl[2];
  read_all(hdr, sizeof(hdr));
  read_all(fl, sizeof(fl));
  const int L = hdr[0], d = hdr[1], hq = hdr[2], hkv = hdr[3], hd = hdr[4], F = hdr[5];
  const int vocab = hdr[6], max_pos = hdr[7], n_chunks = hdr[8], n_query = hdr[9];
  const int ratio_bp = hdr[10];
  if (n_chunks < 1 || n_chunks > 64) die("n_chunks out of range");
  int32_t chunk_len[64];
  read_all(chunk_len, sizeof(int32_t) * (size_t)n_chunks);
  int T = n_query;
  for (int i = 0; i < n_chunks; ++i) T += chunk_len[i];

  cb_model_config cfg = {L, d, hq, hkv, hd, F, vocab, fl[0], fl[1], CB_F32, max_pos};
  cb_layer_weights *lw = (cb_layer_weights *)calloc((size_t)L, sizeof(cb_layer_weights));
  if (!lw) die("out of host memory");
  const void *embed = upload((size_t)vocab * d, sizeof(float));
  const float *final_norm = (const float *)upload((size_t)d, sizeof(float));
  const size_t qkv_rows = (size_t)(hq + 2 * hkv) * hd;
  for (int l = 0; l < L; ++l) {
    lw[l].w_qkv = upload(qkv_rows * d, sizeof(float));
    lw[l].w_o = upload((size_t)d * hq * hd, sizeof(float));
    lw[l].w_gate = upload((size_t)F * d, sizeof(float));
    lw[l].w_up = upload((size_t)F * d, sizeof(float));
    lw[l].w_down = upload((size_t)d * F, sizeof(float));
    lw[l].norm1 = (const float *)upload((size_t)d, sizeof(float));
    lw[l].norm2 = (const float *)upload((size_t)d, sizeof(float));
  }
  const int32_t *tokens = (const int32_t *)upload((size_t)T, sizeof(int32_t));
  fclose(in);

  float *rope = (float *)dev_alloc(cb_rope_table_elems(max_pos, hd) * sizeof(float));
  need(cb_rope_table_init(rope, max_pos, hd, fl[0], NULL), "cb_rope_table_init");
  cb_weights w = {embed, final_norm, lw, rope};
  cb_model *m = NULL;
  need(cb_model_create(&cfg, &w, &m), "cb_model_create");

  /* each chunk prefilled alone at positions 0 .. len - 1 (its PIC cache) */
  const int kvw = hkv * hd;
  cb_segment segs[65];
  int t0 = 0;
  for (int i = 0; i < n_chunks; ++i) {
    const int n = chunk_len[i];
    cb_segment one = {n, NULL, NULL, 0, 0};
    cb_request r = {tokens + t0, &one, 1};
    cb_plan plan;
    need(cb_full_plan(m, &r, 1, &plan), "cb_full_plan");
    void *k = dev_alloc((size_t)L * n * kvw * sizeof(float));
    void *v = dev_alloc((size_t)L * n * kvw * sizeof(float));
    void *ws = dev_alloc(plan.workspace_bytes);
    cb_blend_out o = {k, v, 0, NULL, NULL, NULL, NULL, NULL};
    need(cb_full_prefill(m, &r, 1, &o, ws, plan.workspace_bytes, NULL), "cb_full_prefill");
    segs[i] = (cb_segment){n, k, v, (int64_t)n * kvw, 0};
    t0 += n;
  }
  segs[n_chunks] = (cb_segment){n_query, NULL, NULL, 0, 0};

  /* the request: cached chunks in order, then the query */
  cb_request req = {tokens, segs, n_chunks + 1};
  cb_blend_params p = {0};
  p.ratio_bp = ratio_bp;
  p.policy = CB_POLICY_TOKEN_TOPK;
  p.sel_layer = 1;
  cb_plan plan;
  need(cb_blend_plan(m, &req, 1, &p, &plan), "cb_blend_plan");
  const int K = (int)plan.K_total, R = (int)plan.R_total;
  cb_blend_out o;
  o.k_cache = dev_alloc((size_t)L * plan.T_total * kvw * sizeof(float));
  o.v_cache = dev_alloc((size_t)L * plan.T_total * kvw * sizeof(float));
  o.cache_layer_stride = 0;
  o.deviation = (float *)dev_alloc((size_t)plan.N_total * sizeof(float));
  o.selected = (int32_t *)dev_alloc((size_t)K * sizeof(int32_t));
  o.hidden = (float *)dev_alloc((size_t)R * d * sizeof(float));
  o.rows = (int32_t *)dev_alloc((size_t)R * sizeof(int32_t));
  o.first_token = (int32_t *)dev_alloc(sizeof(int32_t));
  void *ws = dev_alloc(plan.workspace_bytes);
  need(cb_blend_prefill(m, &req, 1, &p, &o, ws, plan.workspace_bytes, NULL), "cb_blend_prefill");
  cuda(cudaDeviceSynchronize(), "synchronize");
  cb_status dev_status;
  need(cb_get_device_status(&dev_status), "cb_get_device_status");
  need(dev_status, "device status");

  int32_t *sel = (int32_t *)malloc((size_t)(K + 1) * sizeof(int32_t));
  int32_t *rows = (int32_t *)malloc((size_t)(R + 1) * sizeof(int32_t));
  float *hidden = (float *)malloc((size_t)R * d * sizeof(float) + 1);
  int32_t first;
  if (!sel || !rows || !hidden) die("out of host memory");
  cuda(cudaMemcpy(sel, o.selected, (size_t)K * sizeof(int32_t), cudaMemcpyDeviceToHost), "read");
  cuda(cudaMemcpy(rows, o.rows, (size_t)R * sizeof(int32_t), cudaMemcpyDeviceToHost), "read");
  cuda(cudaMemcpy(hidden, o.hidden, (size_t)R * d * sizeof(float), cudaMemcpyDeviceToHost),
       "read");
  cuda(cudaMemcpy(&first, o.first_token, sizeof(int32_t), cudaMemcpyDeviceToHost), "read");
  cb_model_destroy(m);

  FILE *out = fopen(argv[2], "wb");
  if (!out) die("cannot open the output file");
  const int32_t head[3] = {K, R, first};
  if (fwrite(head, sizeof(head), 1, out) != 1 ||
      fwrite(sel, sizeof(int32_t), (size_t)K, out) != (size_t)K ||
      fwrite(rows, sizeof(int32_t), (size_t)R, out) != (size_t)R ||
      fwrite(hidden, sizeof(float), (size_t)R * d, out) != (size_t)R * d)
    die("short write");
  fclose(out);
  return 0;
}
