/*
 * Float64 CPU oracle for one Medusa verify step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, calls or
 * includes this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark load it (through oracle/oracle.py).  It shares no header,
 * helper or table with the CUDA path.
 *
 * Every routine is the plain definition written out as loops, single-threaded,
 * in double precision.  bf16 inputs are decoded exactly (a bf16 value is the
 * top 16 bits of an IEEE binary32), fp32 inputs are widened exactly.
 *
 * Sources (page title, section):
 *  - "Medusa: Simple LLM Inference Acceleration Framework with Multiple
 *    Decoding Heads" (review page), section "Medusa 的三个核心组件" (the three
 *    core components): head formula p_t^(k) = softmax(W2 (SiLU(W1 h_t) + h_t)),
 *    the ancestor-only tree mask, and typical acceptance with threshold
 *    min(eps, delta * exp(-H(p))), first token accepted unconditionally,
 *    longest valid prefix kept.
 *  - same page, section "方法细节" (method details): temperature 0 reduces the
 *    typical test to greedy decoding.
 *  - same page, FAQ "树注意力为什么能一次验证多条候选": tree position encoding
 *    (each node is encoded at its position in the tree).
 *  - "Medusa 多解码头推理加速全解析" (skill-pack guide), section "推理算法":
 *    per-head top-k of the head logits, candidate verification with
 *    past_key_values, "accept longest valid candidate".
 *
 * Readings taken where the pages are silent (each is also listed in the design
 * notes): no bias terms; one W1/W2 pair per head; u kept exact (double);
 * top-k ordered by (logit descending, index ascending); attention scale is a
 * caller argument (1/sqrt(d) by default) and q head h reads kv head h / G;
 * entropy uses the natural log of p = softmax(z / T); the typical test is the
 * strict inequality p > threshold; at T == 0 the test is argmax-match; the
 * best node is the deepest accepted node, lowest canonical index on ties; the
 * next root token is the argmax of the base logits at the best node.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* Element i of a buffer of floats (dt == ORC_F32) or bf16 bit patterns. */
static double orc_load(const void* p, int dt, size_t i) {
  if (dt == ORC_F32) return (double)((const float*)p)[i];
  uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* True when (va, ia) ranks ahead of (vb, ib): larger value first, then the
 * lower index. */
static int orc_ahead(double va, int ia, double vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

/*
 * Top-k of one row z[0..n) by repeated selection: pick the best element not
 * yet taken, topk times.  Writes indices and values in rank order.
 */
static void orc_topk_row(const double* z, int n, int topk, int32_t* idx, double* val) {
  char* taken = (char*)calloc((size_t)n, 1);
  for (int r = 0; r < topk; ++r) {
    int best = -1;
    for (int v = 0; v < n; ++v) {
      if (taken[v]) continue;
      if (best < 0 || orc_ahead(z[v], v, z[best], best)) best = v;
    }
    taken[best] = 1;
    idx[r] = best;
    val[r] = z[best];
  }
  free(taken);
}

/*
 * Medusa heads.  For every batch row b and head k:
 *   a_j   = sum_i W1[k][j][i] * h[b][i]
 *   u_j   = SiLU(a_j) + h[b][j],        SiLU(x) = x / (1 + exp(-x))
 *   z_v   = sum_j W2[k][v][j] * u_j
 * then the top-k of z (softmax is monotone, so ranking logits ranks p).
 * Layouts: h [B][H], W1 [K][H][H] (out, in), W2 [K][V][H] (vocab, in),
 * u_out [B][K][H] (may be NULL), z_out [B][K][V] (may be NULL),
 * idx/val [B][K][topk].
 */
int orc_heads(const void* h, const void* w1, const void* w2, int dt, int B, int H, int V, int K,
              int topk, double* u_out, double* z_out, int32_t* idx, double* val) {
  if (B < 0 || H <= 0 || V <= 0 || K <= 0 || topk <= 0 || topk > V) return 1;
  double* u = (double*)malloc(sizeof(double) * (size_t)H);
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  if (!u || !z) { free(u); free(z); return 2; }
  for (int b = 0; b < B; ++b) {
    for (int k = 0; k < K; ++k) {
      for (int j = 0; j < H; ++j) {
        double a = 0.0;
        for (int i = 0; i < H; ++i)
          a += orc_load(w1, dt, ((size_t)k * H + j) * H + i) * orc_load(h, dt, (size_t)b * H + i);
        u[j] = a / (1.0 + exp(-a)) + orc_load(h, dt, (size_t)b * H + j);
      }
      for (int v = 0; v < V; ++v) {
        double s = 0.0;
        for (int j = 0; j < H; ++j) s += orc_load(w2, dt, ((size_t)k * V + v) * H + j) * u[j];
        z[v] = s;
      }
      size_t bk = (size_t)b * K + k;
      if (u_out) memcpy(u_out + bk * H, u, sizeof(double) * (size_t)H);
      if (z_out) memcpy(z_out + bk * V, z, sizeof(double) * (size_t)V);
      orc_topk_row(z, V, topk, idx + bk * topk, val + bk * topk);
    }
  }
  free(u);
  free(z);
  return 0;
}

/* Top-k of each of `rows` rows of fp32 values (the ranking step alone). */
int orc_topk_f32(const float* x, int rows, int n, int topk, int32_t* idx, double* val) {
  if (rows < 0 || n <= 0 || topk <= 0 || topk > n) return 1;
  double* z = (double*)malloc(sizeof(double) * (size_t)n);
  if (!z) return 2;
  for (int r = 0; r < rows; ++r) {
    for (int v = 0; v < n; ++v) z[v] = (double)x[(size_t)r * n + v];
    orc_topk_row(z, n, topk, idx + (size_t)r * topk, val + (size_t)r * topk);
  }
  free(z);
  return 0;
}

/*
 * Tree attention.  For layer l, batch row b, node i and q head hq, with
 * G = Hq / Hkv and kv head g = hq / G, the keys visible to node i are the
 * prefix rows 0..L_b-1 of the cache and the tree rows j whose bit (i, j) is
 * set in the ancestor mask (ancestors and the node itself):
 *   s_j = scale * <q, k_j>,   out = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m)
 * Layouts: q [nl][B][N][Hq][d]; kc, vc [nl][B][Lmax][Hkv][d];
 * kt, vt [nl][B][N][Hkv][d]; mask [N][ceil(N/32)] (bit j%32 of word j/32);
 * out [nl][B][N][Hq][d].
 */
int orc_tree_attention(const void* q, const void* kc, const void* vc, const void* kt,
                       const void* vt, int dt, const uint32_t* mask, const int32_t* prefix_len,
                       int nl, int B, int N, int Hq, int Hkv, int d, int Lmax, double scale,
                       double* out) {
  if (nl <= 0 || B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return 1;
  int G = Hq / Hkv, W = (N + 31) / 32;
  for (int b = 0; b < B; ++b)
    if (prefix_len[b] < 0 || prefix_len[b] > Lmax) return 1;
  double* s = (double*)malloc(sizeof(double) * (size_t)(Lmax + N));
  char* vis = (char*)malloc((size_t)(Lmax + N));
  if (!s || !vis) { free(s); free(vis); return 2; }
  for (int l = 0; l < nl; ++l)
    for (int b = 0; b < B; ++b) {
      int L = prefix_len[b];
      for (int i = 0; i < N; ++i)
        for (int hq = 0; hq < Hq; ++hq) {
          int g = hq / G;
          size_t qo = ((((size_t)l * B + b) * N + i) * Hq + hq) * d;
          double m = -INFINITY;
          for (int j = 0; j < L + N; ++j) {
            const void* kb;
            size_t ko;
            if (j < L) {
              vis[j] = 1;
              kb = kc;
              ko = ((((size_t)l * B + b) * Lmax + j) * Hkv + g) * d;
            } else {
              int t = j - L;
              vis[j] = (char)((mask[(size_t)i * W + t / 32] >> (t % 32)) & 1u);
              kb = kt;
              ko = ((((size_t)l * B + b) * N + t) * Hkv + g) * d;
            }
            if (!vis[j]) continue;
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += orc_load(q, dt, qo + c) * orc_load(kb, dt, ko + c);
            s[j] = scale * acc;
            if (s[j] > m) m = s[j];
          }
          double den = 0.0;
          double* o = out + qo;
          for (int c = 0; c < d; ++c) o[c] = 0.0;
          for (int j = 0; j < L + N; ++j) {
            if (!vis[j]) continue;
            double w = exp(s[j] - m);
            den += w;
            const void* vb;
            size_t vo;
            if (j < L) {
              vb = vc;
              vo = ((((size_t)l * B + b) * Lmax + j) * Hkv + g) * d;
            } else {
              vb = vt;
              vo = ((((size_t)l * B + b) * N + (j - L)) * Hkv + g) * d;
            }
            for (int c = 0; c < d; ++c) o[c] += w * orc_load(vb, dt, vo + c);
          }
          for (int c = 0; c < d; ++c) o[c] /= den;
        }
    }
  free(s);
  free(vis);
  return 0;
}

/*
 * Statistics of the base distribution at one tree node, from its fp32 logits
 * z[0..V): the argmax (lowest index on ties), and for T > 0 the tempered
 * distribution p_v = exp(z_v / T) / sum exp(z_u / T) (evaluated as
 * exp((z_v - max) / T) for range), its entropy H = -sum p ln p, and the typical
 * threshold min(eps, delta * exp(-H)).  At T == 0 the distribution is the
 * one-hot limit, so H = 0 and the threshold is min(eps, delta).
 */
static void orc_node_stats(const float* z, int V, double T, double eps, double delta, int* amax,
                           double* zmax, double* sum, double* thr) {
  int a = 0;
  for (int v = 1; v < V; ++v)
    if (z[v] > z[a]) a = v;
  *amax = a;
  *zmax = (double)z[a];
  if (T == 0.0) {
    *sum = 1.0;
    *thr = eps < delta ? eps : delta;
    return;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) S += exp(((double)z[v] - *zmax) / T);
  double H = 0.0;
  for (int v = 0; v < V; ++v) {
    double p = exp(((double)z[v] - *zmax) / T) / S;
    if (p > 0.0) H -= p * log(p);
  }
  double e = delta * exp(-H);
  *sum = S;
  *thr = eps < e ? eps : e;
}

/*
 * Typical acceptance over one candidate tree per batch row.
 * logits [B][N][V] fp32: the base model's next-token logits at every node.
 * tokens [B][N]: node tokens (node 0 is the root).  parent [N]: parent index,
 * parent[0] = -1, parent[n] < n.
 * Node n >= 1 passes its test when p_parent(tokens[n]) > thr_parent (T > 0) or
 * tokens[n] == argmax of the parent's logits (T == 0).  The root is accepted
 * unconditionally; accepted(n) = accepted(parent(n)) and test(n).  The best node
 * is the deepest accepted node (lowest index on ties); path_nodes[b] lists root
 * to best, padded with -1 up to Dmax + 1 entries; accept_len = depth(best) + 1;
 * next_tok = argmax of the logits at the best node.
 * Optional outputs (may be NULL): p_tok [B][N] (probability the parent gives the
 * node's token; 1 at the root), thr [B][N] (the parent's threshold; 0 at the
 * root), accepted [B][N] (0/1).
 */
int orc_typical_accept(const float* logits, const int32_t* tokens, const int32_t* parent, int B,
                       int N, int V, double T, double eps, double delta, int Dmax,
                       int32_t* accept_len, int32_t* path_nodes, int32_t* next_tok, double* p_tok,
                       double* thr, uint8_t* accepted) {
  if (B < 0 || N <= 0 || V <= 0 || T < 0.0 || parent[0] != -1) return 1;
  for (int n = 1; n < N; ++n)
    if (parent[n] < 0 || parent[n] >= n) return 1;
  int* depth = (int*)malloc(sizeof(int) * (size_t)N);
  int* amax = (int*)malloc(sizeof(int) * (size_t)N);
  double* zmax = (double*)malloc(sizeof(double) * (size_t)N);
  double* S = (double*)malloc(sizeof(double) * (size_t)N);
  double* th = (double*)malloc(sizeof(double) * (size_t)N);
  uint8_t* acc = (uint8_t*)malloc((size_t)N);
  depth[0] = 0;
  int deepest = 0;
  for (int n = 1; n < N; ++n) {
    depth[n] = depth[parent[n]] + 1;
    if (depth[n] > deepest) deepest = depth[n];
  }
  if (deepest > Dmax) {
    free(depth); free(amax); free(zmax); free(S); free(th); free(acc);
    return 1;
  }
  for (int b = 0; b < B; ++b) {
    for (int n = 0; n < N; ++n)
      orc_node_stats(logits + ((size_t)b * N + n) * V, V, T, eps, delta, &amax[n], &zmax[n], &S[n],
                     &th[n]);
    acc[0] = 1;
    if (p_tok) p_tok[(size_t)b * N] = 1.0;
    if (thr) thr[(size_t)b * N] = 0.0;
    for (int n = 1; n < N; ++n) {
      int par = parent[n];
      int x = tokens[(size_t)b * N + n];
      int test;
      double p;
      if (T == 0.0) {
        test = (x == amax[par]);
        p = test ? 1.0 : 0.0;
      } else {
        double zx = (double)logits[((size_t)b * N + par) * V + x];
        p = exp((zx - zmax[par]) / T) / S[par];
        test = p > th[par];
      }
      acc[n] = (uint8_t)(acc[par] && test);
      if (p_tok) p_tok[(size_t)b * N + n] = p;
      if (thr) thr[(size_t)b * N + n] = th[par];
    }
    int best = 0;
    for (int n = 1; n < N; ++n)
      if (acc[n] && depth[n] > depth[best]) best = n;
    for (int i = 0; i <= Dmax; ++i) path_nodes[(size_t)b * (Dmax + 1) + i] = -1;
    for (int n = best; n >= 0; n = parent[n]) path_nodes[(size_t)b * (Dmax + 1) + depth[n]] = n;
    accept_len[b] = depth[best] + 1;
    next_tok[b] = amax[best];
    if (accepted) memcpy(accepted + (size_t)b * N, acc, (size_t)N);
  }
  free(depth); free(amax); free(zmax); free(S); free(th); free(acc);
  return 0;
}

/*
 * KV compaction: for each batch row b, the accepted path's tree rows are
 * appended to the cache after the prefix:
 *   kc[l][b][L_b + i] = kt[l][b][path_nodes[b][i]]  for i < accept_len[b]
 * (same for v), new_len[b] = L_b + accept_len[b].  A row whose append would
 * pass Lmax is left untouched and reported in overflow[b] = 1.
 * Rows are copied as raw bytes (elem_bytes per element).
 */
int orc_kv_compact(void* kc, void* vc, const void* kt, const void* vt, int elem_bytes,
                   const int32_t* path_nodes, const int32_t* accept_len, const int32_t* prefix_len,
                   int32_t* new_len, int32_t* overflow, int nl, int B, int N, int Hkv, int d,
                   int Lmax, int Dmax) {
  size_t row = (size_t)Hkv * d * elem_bytes;
  for (int b = 0; b < B; ++b) {
    int L = prefix_len[b], A = accept_len[b];
    if (A < 1 || A > Dmax + 1) return 1;
    if (L + A > Lmax) {
      overflow[b] = 1;
      new_len[b] = L;
      continue;
    }
    overflow[b] = 0;
    for (int l = 0; l < nl; ++l)
      for (int i = 0; i < A; ++i) {
        int src = path_nodes[(size_t)b * (Dmax + 1) + i];
        if (src < 0 || src >= N) return 1;
        size_t so = (((size_t)l * B + b) * N + src) * row;
        size_t dof = (((size_t)l * B + b) * Lmax + L + i) * row;
        memcpy((char*)kc + dof, (const char*)kt + so, row);
        memcpy((char*)vc + dof, (const char*)vt + so, row);
      }
    new_len[b] = L + A;
  }
  return 0;
}

/*
 * Rotary position embedding of the tree tokens at their tree positions.
 * Review page, FAQ "树注意力为什么能一次验证多条候选": position encoding follows
 * the tree, so node n of row b sits at pos[b][n] = prefix_len[b] + depth(n)
 * (the positions medusa tree packing produces).  The pages give no formula;
 * reading: the rotate-half rotary embedding of the LLaMA family (Vicuna is
 * one): for i < d/2 the pair (x[i], x[i + d/2]) is rotated by the angle
 * pos * theta_i, theta_i = base^(-2i/d):
 *   x'[i]       = x[i] cos(a) - x[i + d/2] sin(a)
 *   x'[i + d/2] = x[i + d/2] cos(a) + x[i] sin(a),   a = pos * theta_i.
 * x [nl][B][N][Hx][d] (fp32 or bf16 bits) -> out (same layout) in double.
 */
int orc_tree_rope(const void* x, int dt, const int32_t* pos, int nl, int B, int N, int Hx, int d, double base,
                  double* out) {
  if (d < 2 || d % 2 || base <= 0.0) return 1;
  const int half = d / 2;
  for (int l = 0; l < nl; ++l)
    for (int b = 0; b < B; ++b)
      for (int n = 0; n < N; ++n) {
        const double p = (double)pos[(size_t)b * N + n];
        for (int h = 0; h < Hx; ++h) {
          const size_t o = ((((size_t)l * B + b) * N + n) * Hx + h) * d;
          for (int i = 0; i < half; ++i) {
            const double a = p * pow(base, -2.0 * i / d);
            const double x0 = orc_load(x, dt, o + i), x1 = orc_load(x, dt, o + i + half);
            out[o + i] = x0 * cos(a) - x1 * sin(a);
            out[o + i + half] = x1 * cos(a) + x0 * sin(a);
          }
        }
      }
  return 0;
}

/*
 * Medusa-1 head loss and its gradient with respect to the head logits.
 * Review page, section "方法细节" (training recipe): with the backbone frozen,
 * only the heads train, on L1 = -sum_{k=1..K} lambda_k log p_t^(k)(y_{t+k+1}),
 * lambda_k = 0.8^k (here decay^k): head k, read at position t, is scored on
 * the token k + 1 places ahead.
 *
 * Readings: the loss of head k is the mean over the counted positions of the
 * batch (the mean cross entropy of the guide's training loop, "Medusa 多解码头
 * 推理加速全解析", training section), and L1 is the lambda-weighted sum of
 * these means.  Position t of sequence b counts for head k when t + k + 1 < S
 * and its target y[b][t+k+1] is not negative (a negative target marks padding
 * and is skipped); a head with no counted position has loss 0.
 *
 * logits [K][B][S][V] (fp32 or bf16 bits), head k stored at index k - 1;
 * tokens [B][S].  Outputs: counts[K] (n_k), loss[K + 1] (the K means, then
 * L1), row_loss[K][B][S] (-log p of the target, 0 where not counted) and, when
 * dlogits is not NULL, dL1/dz = lambda_k / n_k * (softmax(z) - onehot(y)) on
 * counted rows, 0 elsewhere.  counts_in, when not NULL, replaces the counts as
 * the normaliser (a slice of sequences cut from a larger batch).
 * Returns 2 when a target is >= V.
 */
int orc_head_loss(const void* logits, int dt, const int32_t* tokens, int K, int B, int S, int V, double decay,
                  const int32_t* counts_in, int32_t* counts, double* loss, double* row_loss, double* dlogits) {
  if (K < 1 || B < 1 || S < 1 || V < 1) return 1;
  for (size_t i = 0; i < (size_t)B * S; ++i)
    if (tokens[i] >= V) return 2;
  for (int k = 1; k <= K; ++k) {
    int n = 0;
    for (int b = 0; b < B; ++b)
      for (int t = 0; t + k + 1 < S; ++t)
        if (tokens[(size_t)b * S + t + k + 1] >= 0) ++n;
    counts[k - 1] = counts_in ? counts_in[k - 1] : n;
  }
  double* row = (double*)malloc(sizeof(double) * (size_t)V);
  if (!row) return 1;
  double total = 0.0;
  for (int k = 1; k <= K; ++k) {
    const double lambda = pow(decay, (double)k);
    const int n = counts[k - 1];
    double sum = 0.0;
    for (int b = 0; b < B; ++b)
      for (int t = 0; t < S; ++t) {
        const size_t r = ((size_t)(k - 1) * B + b) * S + t;
        const int y = t + k + 1 < S ? tokens[(size_t)b * S + t + k + 1] : -1;
        double* g = dlogits ? dlogits + r * V : NULL;
        if (y < 0 || n <= 0) {
          row_loss[r] = 0.0;
          if (g) memset(g, 0, sizeof(double) * (size_t)V);
          continue;
        }
        double m = -INFINITY;
        for (int v = 0; v < V; ++v) {
          row[v] = orc_load(logits, dt, r * V + v);
          if (row[v] > m) m = row[v];
        }
        double s = 0.0;
        for (int v = 0; v < V; ++v) s += exp(row[v] - m);
        const double lse = m + log(s);
        row_loss[r] = lse - row[y];
        sum += row_loss[r];
        if (g)
          for (int v = 0; v < V; ++v) g[v] = lambda / n * (exp(row[v] - lse) - (v == y ? 1.0 : 0.0));
      }
    loss[k - 1] = n > 0 ? sum / n : 0.0;
    total += lambda * loss[k - 1];
  }
  loss[K] = total;
  free(row);
  return 0;
}
