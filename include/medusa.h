/*
 * medusa.h — C ABI of libmedusa_gb300.so: one Medusa verify step on one GPU.
 *
 * The step (paper review "Medusa: Simple LLM Inference Acceleration Framework
 * with Multiple Decoding Heads", section "Medusa 的三个核心组件"): the Medusa
 * heads propose candidates, the candidates are packed into one tree and
 * verified in a single tree-attention pass, typical acceptance keeps the
 * longest valid prefix, and the accepted tokens' keys/values are appended to
 * the cache.
 *
 * Conventions shared by every compute call:
 *  - Every tensor argument is a caller-owned DEVICE pointer to a dense,
 *    row-major array in the layout stated at the call.  The library never
 *    allocates, frees or retains memory; scratch comes from a caller buffer
 *    sized by the matching *_workspace_size() query (NULL/0 when it returns 0).
 *  - Every compute call is stream-ordered: it validates its arguments on the
 *    host, enqueues kernels on `stream` and returns without synchronising.
 *    Data-dependent results (accept lengths, cache lengths) stay on the
 *    device, so a whole step can be captured in a CUDA graph.
 *  - Host-side validation failures return a medusa_status without launching.
 *  - Errors only the device can see (an index out of range, a cache overflow,
 *    a malformed topology) are recorded in the caller's int32 device word
 *    `d_status` (first error wins, 0 = none); medusa_status_check() reads it.
 *    `d_status` may be NULL, in which case device errors are not reported
 *    (the offending element is still skipped, never written out of bounds).
 *  - The library never aborts, prints or traps.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).
 */
#ifndef MEDUSA_GB300_H
#define MEDUSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* medusa_stream_t; /* identical to cudaStream_t */

typedef enum medusa_status {
  MEDUSA_OK = 0,
  MEDUSA_ERR_INVALID_ARG = 1, /* a size, pointer or value outside its stated range */
  MEDUSA_ERR_UNSUPPORTED = 2, /* valid, but no kernel of this build handles it */
  MEDUSA_ERR_ALIAS = 3,       /* buffers that must not overlap do */
  MEDUSA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, copy, attribute) */
  MEDUSA_ERR_WORKSPACE = 5    /* workspace NULL or smaller than the query returned */
} medusa_status;

typedef enum medusa_dtype {
  MEDUSA_F32 = 0, /* IEEE binary32 */
  MEDUSA_BF16 = 1 /* bfloat16 (upper half of binary32) */
} medusa_dtype;

/* Codes written to d_status by device code. */
#define MEDUSA_DEV_OK 0
#define MEDUSA_DEV_BAD_INDEX 1      /* a token, rank or node index outside its range */
#define MEDUSA_DEV_CACHE_OVERFLOW 2 /* prefix_len + accept_len would pass Lmax */
#define MEDUSA_DEV_TIMEOUT 3        /* a bounded device-side wait gave up */
#define MEDUSA_DEV_BAD_TOPOLOGY 4   /* parent[n] >= n, or depth inconsistent */
#define MEDUSA_DEV_BAD_LENGTH 5     /* prefix_len outside [0, Lmax] */

#define MEDUSA_MAX_NODES 256 /* tree nodes including the root */
#define MEDUSA_MAX_DEPTH 16  /* tree depth = number of Medusa heads used */
#define MEDUSA_MAX_TOPK 32   /* candidates kept per head */

/* ------------------------------------------------------------------ topology
 * A candidate tree (skill-pack guide "Medusa 多解码头推理加速全解析", sections
 * "候选生成" and "树结构：medusa_choices"; paper review, "方法细节", sparse tree).
 * A node is named by its rank path: element j is the rank, within Medusa head
 * j+1's top-k list, of the token at depth j+1 (the medusa_choices format).
 * Canonical order: paths sorted by (length, lexicographic); node 0 is the
 * root (empty path) and every parent precedes its children.
 */
typedef struct medusa_topology {
  int32_t n_nodes;   /* 1..MEDUSA_MAX_NODES, root included */
  int32_t max_depth; /* deepest node's depth (root = 0) */
  int32_t n_leaves;  /* nodes without children */
  int32_t max_rank;  /* 1 + largest rank used: the heads must keep at least this many */
  int32_t parent[MEDUSA_MAX_NODES]; /* parent[0] = -1, parent[n] < n */
  int32_t depth[MEDUSA_MAX_NODES];
  int32_t rank[MEDUSA_MAX_NODES];   /* rank within head depth-1's top-k; -1 at the root */
  int32_t retrieve[MEDUSA_MAX_NODES * (MEDUSA_MAX_DEPTH + 1)];
  /* retrieve[leaf * (max_depth+1) + j]: node at depth j on the path root..leaf
   * (leaves in canonical order), -1 past the leaf. */
} medusa_topology;

/* Device-resident copy of a topology (pointers into a caller-owned buffer). */
typedef struct medusa_dev_topology {
  int32_t n_nodes, max_depth, n_leaves, max_rank;
  const int32_t* parent;   /* [n_nodes] */
  const int32_t* depth;    /* [n_nodes] */
  const int32_t* rank;     /* [n_nodes] */
  const int32_t* retrieve; /* [n_leaves][max_depth+1] */
} medusa_dev_topology;

/* Tree from an explicit medusa_choices list.  `ranks` holds all paths back to
 * back, `path_len[i]` the length of path i (>= 1).  The root is added,
 * duplicates are dropped, every path's parent must be present.  Host only.
 * INVALID_ARG on a negative rank, a missing parent, a path longer than
 * MEDUSA_MAX_DEPTH or more than max_nodes nodes. */
medusa_status medusa_topology_from_paths(const int32_t* ranks, const int32_t* path_len,
                                         int n_paths, int max_nodes, medusa_topology* out);

/* Dense Cartesian tree (guide, "候选生成": itertools.product over the heads'
 * top-k lists): depth j+1 takes ranks < topk_per_head[j], j < K; canonical
 * order, truncated to max_nodes (root counted).  Host only. */
medusa_status medusa_topology_dense(int K, const int32_t* topk_per_head, int max_nodes,
                                    medusa_topology* out);

/* Greedy sparse tree (paper review, "方法细节": calibration top-i accuracies,
 * nodes chosen greedily by expected-acceptance gain).  acc[k*R + i] is head
 * k's top-(i+1) accuracy (k, i 0-based).  A node's gain is the probability it
 * is reached, prod_j acc[j][r_j]; the frontier node with the largest gain is
 * added until n_nodes nodes (root counted).  Gains within a relative 1e-12 are
 * ties, broken by the shallower path, then the lexicographically smaller one.
 * Host only. */
medusa_status medusa_topology_greedy(const double* acc, int K, int R, int n_nodes,
                                     medusa_topology* out);

/* Number of int32 elements medusa_topology_upload() needs in its buffer. */
size_t medusa_topology_device_elems(const medusa_topology* t);

/* Copies `t` into the caller's device buffer `d_buf` (>= the elems above) and
 * fills `out` with pointers into it.  Synchronous set-up call: returns once the
 * copy is done, so `t` may be freed afterwards. */
medusa_status medusa_topology_upload(const medusa_topology* t, int32_t* d_buf, size_t buf_elems,
                                     medusa_dev_topology* out, medusa_stream_t stream);

/* -------------------------------------------------------------- (a) heads
 * Medusa heads on the last hidden state (paper review, "Medusa 的三个核心组件":
 * p^(k) = softmax(W2^(k) (SiLU(W1^(k) h) + h)); guide, "候选生成": top-k per
 * head).  For every row b and head k:
 *   u = SiLU(W1[k] h[b]) + h[b]   (fp32),   z = W2[k] u   (fp32 accumulation)
 * and the top-k of z, ranked (logit descending, index ascending); softmax is
 * monotone, so ranking logits ranks probabilities.
 *   h          [B][H]        dtype dt
 *   w1         [K][H][H]     dtype dt, row = output unit, column = input unit
 *   w2         [K][V][H]     dtype dt, row = vocabulary entry
 *   topk_idx   [B][K][topk]  int32 out
 *   topk_logit [B][K][topk]  fp32 out
 *   logits_or_null [B][K][V] fp32 out, optional (all head logits z)
 * 1 <= B <= 64, 1 <= K <= MEDUSA_MAX_DEPTH, 1 <= topk <= min(V, MEDUSA_MAX_TOPK),
 * H a multiple of 8, pointers 16-byte aligned.  bf16 batches of 4 to 64 with H
 * a multiple of 64 run both passes on tcgen05 tensor cores (the fp32 u split
 * into bf16 hi + lo operands); smaller batches and fp32 stream the weights on
 * CUDA cores.  The workspace holds u, the logits z when logits_or_null is NULL
 * and the top-k candidate lists. */
size_t medusa_heads_workspace_size(int B, int H, int V, int K, int topk);
medusa_status medusa_heads(const void* h, const void* w1, const void* w2, int B, int H, int V,
                           int K, int topk, medusa_dtype dt, int32_t* topk_idx, float* topk_logit,
                           float* logits_or_null, void* ws, size_t ws_bytes, int32_t* d_status,
                           medusa_stream_t stream);

/* The ranking step of medusa_heads alone: top-k of each of `rows` fp32 rows
 * of length V (logits [rows][V]), ranked (value descending, index ascending).
 * Same limits on topk. */
size_t medusa_head_topk_workspace_size(int rows, int V, int topk);
medusa_status medusa_head_topk(const float* logits, int rows, int V, int topk, int32_t* topk_idx,
                               float* topk_logit, void* ws, size_t ws_bytes,
                               medusa_stream_t stream);

/* ---------------------------------------------------------- (b) tree_build
 * Packs the candidate tree of every batch row (guide, "树形注意力" and
 * "候选生成"; paper review FAQ, "位置编码按树结构调整": positions follow the tree).
 *   tokens[b][0] = root_tok[b];  tokens[b][n] = topk_idx[b][depth(n)-1][rank(n)]
 *   pos[b][n]    = prefix_len[b] + depth(n)
 *   mask[n][w]   bit (j % 32) of word j / 32 set iff node j is n or an ancestor
 *                of n (batch-independent, ceil(N/32) words per node); mask may be
 *                NULL: it depends on the topology alone, so a caller that holds it
 *                for this topology can skip it (the topology checks still run)
 *   root_tok [B], prefix_len [B], tokens [B][N], pos [B][N]: int32;
 *   topk_idx [B][K][topk] from medusa_heads.  Needs topology max_depth <= K and
 *   max_rank <= topk (INVALID_ARG otherwise).  A rank or parent that the device
 *   finds out of range sets BAD_INDEX / BAD_TOPOLOGY and writes -1 there. */
medusa_status medusa_tree_build(const medusa_dev_topology* t, const int32_t* root_tok,
                                const int32_t* topk_idx, int B, int K, int topk,
                                const int32_t* prefix_len, int32_t* tokens, int32_t* pos,
                                uint32_t* mask, int32_t* d_status, medusa_stream_t stream);

/* ------------------------------------------------------ (c) tree_attention
 * Tree attention (paper review, "Medusa 的三个核心组件": each token attends only
 * to its own branch's predecessors; FAQ: one pass verifies every candidate and
 * reuses the common prefix; guide, "树形验证": verification with
 * past_key_values).  For layer l, row b, node i, q head h (G = Hq / Hkv, kv
 * head g = h / G): keys = prefix cache rows 0..prefix_len[b]-1 plus the tree
 * rows j with mask bit (i, j) set;
 *   out = softmax(scale * q K^T) V   (fp32 accumulation and softmax)
 *   q   [n_layers][B][N][Hq][d]      kc, vc [n_layers][B][Lmax][Hkv][d]
 *   kt, vt [n_layers][B][N][Hkv][d]  mask [N][ceil(N/32)] from tree_build
 *   prefix_len [B]                   out [n_layers][B][N][Hq][d] (dtype dt)
 * All layers are processed in one call.  bf16 with d == 128 and 128 % G == 0
 * runs on the tcgen05 tensor-core kernel (TMA-staged K/V tiles, TMEM
 * accumulators); other shapes and fp32 run on CUDA cores (fp32 FFMA; fp32
 * never uses TF32).  Cache rows at and past prefix_len[b] are never read into
 * the result.  prefix_len outside [0, Lmax] sets BAD_LENGTH and the row's
 * output is left unwritten.  Limits: N <= MEDUSA_MAX_NODES, d a multiple of 32,
 * d <= 256, Hq a multiple of Hkv, pointers 16-byte aligned.
 * Split key ranges: the tensor-core kernel runs whole (layer, row, kv-head
 * group) items in full rounds over the SMs; when the last round would leave
 * SMs idle, each of its items is split into key-range pieces whose partial
 * results (unnormalised O, row maximum, row sum) are merged by a second kernel
 * in the same call (online-softmax rescaling).  The partials need
 * medusa_tree_attention_workspace_size() bytes of 16-byte aligned workspace
 * (0 when no split is planned for these sizes on the current device). */
size_t medusa_tree_attention_workspace_size(int n_layers, int B, int N, int Hq, int Hkv, int d,
                                            int Lmax, medusa_dtype dt);
medusa_status medusa_tree_attention(const void* q, const void* kc, const void* vc, const void* kt,
                                    const void* vt, const uint32_t* mask,
                                    const int32_t* prefix_len, int n_layers, int B, int N, int Hq,
                                    int Hkv, int d, int Lmax, float scale, medusa_dtype dt,
                                    void* out, void* ws, size_t ws_bytes, int32_t* d_status,
                                    medusa_stream_t stream);

/* ------------------------------------------------------ (d) typical_accept
 * Typical acceptance (paper review, "Medusa 的三个核心组件": a candidate passes
 * when its probability exceeds min(eps, delta * exp(-H(p))), the first token
 * is accepted greedily and unconditionally, the longest valid prefix is kept;
 * "方法细节": temperature 0 reduces to greedy decoding; guide, "树形验证":
 * "accept longest valid candidate").
 *   logits [B][N][V] fp32: base logits at every tree node (what the backbone
 *   predicts after that node).  p = softmax(logits / temperature), H = -sum p ln p.
 *   Node n >= 1 passes when p_parent(tokens[b][n]) > min(eps, delta*exp(-H_parent))
 *   (temperature > 0) or tokens[b][n] == argmax of the parent's logits
 *   (temperature == 0).  accepted(root) = 1; accepted(n) = accepted(parent) and
 *   pass(n).  Best node = deepest accepted node, lowest index on ties.
 *   accept_len [B] = depth(best) + 1 (1 .. max_depth+1)
 *   path_nodes [B][max_depth+1] = node indices root..best, -1 after
 *   next_tok [B] = argmax of the best node's logits (lowest index on ties)
 *   p_tok_or_null, thr_or_null [B][N]: the probability the parent gives the
 *   node's token and the parent's threshold (root: 1 and 0), optional.
 *   tokens [B][N] int32 from tree_build; token ids must lie in [0, V) (else
 *   BAD_INDEX and the node fails its test).  temperature >= 0, eps >= 0,
 *   delta >= 0.  The workspace (16-byte aligned) holds per-chunk partial
 *   statistics of every node's logit row. */
size_t medusa_typical_accept_workspace_size(int B, int N, int V);
medusa_status medusa_typical_accept(const float* logits, const int32_t* tokens,
                                    const medusa_dev_topology* t, int B, int V, float temperature,
                                    float eps, float delta, int32_t* accept_len,
                                    int32_t* path_nodes, int32_t* next_tok, float* p_tok_or_null,
                                    float* thr_or_null, void* ws, size_t ws_bytes,
                                    int32_t* d_status, medusa_stream_t stream);

/* Allocation-free variant of medusa_typical_accept (the paper has no
 * counterpart; this is a property of the library, not of the method).
 * For callers that cannot allocate device memory where they run the step: a
 * serving loop whose device memory was handed out at start-up (typically to
 * the KV cache), a plugin living under a host framework that owns every
 * allocation, or a latency-critical path that must not enter the CUDA
 * allocator.  Same arguments, results and device error codes as
 * medusa_typical_accept, minus the workspace: the per-chunk statistics go to
 * one static device array of MEDUSA_ACCEPT_NOALLOC_MAX_BYTES that every GPU
 * loading this library holds until the process exits.
 *  - Limit: medusa_typical_accept_workspace_size(B, N, V) must not exceed
 *    MEDUSA_ACCEPT_NOALLOC_MAX_BYTES (1 MiB; e.g. B * N <= 4096 at V = 32000),
 *    else MEDUSA_ERR_UNSUPPORTED before any launch.
 *  - Every call looks up the array's device address in the current context
 *    (a runtime query; MEDUSA_ERR_CUDA if it fails).  The first call in a
 *    context may load the library's device code, and that load is what
 *    allocates the array: make the first call at start-up, before any stream
 *    capture on that device (or load modules eagerly, CUDA_MODULE_LOADING=EAGER).
 *  - Every call on a device uses the same array and leaves its contents
 *    behind; each call writes every entry it reads first, so nothing needs
 *    clearing.  Calls whose kernels overlap on the GPU (different streams
 *    without ordering) race on the array: order them.
 *  - Calls no cudaMalloc / cudaFree or other allocating routine. */
#define MEDUSA_ACCEPT_NOALLOC_MAX_BYTES (1u << 20)
medusa_status medusa_typical_accept_noalloc(const float* logits, const int32_t* tokens,
                                            const medusa_dev_topology* t, int B, int V,
                                            float temperature, float eps, float delta,
                                            int32_t* accept_len, int32_t* path_nodes,
                                            int32_t* next_tok, float* p_tok_or_null,
                                            float* thr_or_null, int32_t* d_status,
                                            medusa_stream_t stream);

/* ----------------------------------------------------------- (e) kv_compact
 * Appends the accepted path's keys/values to the cache (guide, "树形验证":
 * verification with past_key_values and use_cache):
 *   kc[l][b][prefix_len[b] + i] = kt[l][b][path_nodes[b][i]]   i < accept_len[b]
 *   (same for vc/vt), new_len[b] = prefix_len[b] + accept_len[b].
 * Layouts as in tree_attention; path_nodes [B][Dmax+1].  kt/vt must not overlap
 * kc/vc (ALIAS).  new_len may alias prefix_len.  A row whose append would pass
 * Lmax writes nothing, keeps new_len = prefix_len and sets CACHE_OVERFLOW; an
 * accept_len outside 1..Dmax+1 or a path node outside [0, N) sets BAD_INDEX and
 * that row writes nothing. */
medusa_status medusa_kv_compact(void* kc, void* vc, const void* kt, const void* vt,
                                const int32_t* path_nodes, const int32_t* accept_len,
                                const int32_t* prefix_len, int32_t* new_len, int n_layers, int B,
                                int N, int Hkv, int d, int Lmax, int Dmax, medusa_dtype dt,
                                int32_t* d_status, medusa_stream_t stream);

/* ------------------------------------------------------------- (f) tree_rope
 * Rotary position embedding of the verify pass's tree tokens at their tree
 * positions, in place (paper review, FAQ "树注意力为什么能一次验证多条候选":
 * the position encoding follows the tree; pos from medusa_tree_build is
 * prefix_len + depth).  The step just before medusa_tree_attention: q is the
 * verify pass's query tensor and k the tree K buffer (the backbone's key
 * projection of the tree tokens, before rotation), in the layouts of
 * medusa_tree_attention:
 *   q [nl][B][N][Hq][d], k [nl][B][N][Hkv][d] (or NULL: q only), pos [B][N].
 * For i < d/2 the pair (x[i], x[i + d/2]) of every head is rotated by the
 * angle pos[b][n] * base^(-2i/d) (the rotate-half convention of the LLaMA
 * family; the pages give no formula, base 10000 for Vicuna).  Angles are
 * formed and reduced in double precision, the rotation runs in fp32, values
 * are read and written in `dt`.  d even, 2 <= d <= 256; q and k must not
 * overlap (ALIAS).  No device-side errors. */
medusa_status medusa_tree_rope(void* q, void* k, const int32_t* pos, int n_layers, int B, int N, int Hq,
                               int Hkv, int d, float base, medusa_dtype dt, medusa_stream_t stream);

/* ---------------------------------------------------------------- (g) linear
 * One linear layer of the verify pass over the tree tokens (paper review,
 * roofline in "实验设计与结果" and "局限性": verifying N candidates runs every
 * linear layer of the backbone over B * N tokens, which lifts decoding's
 * operational intensity; past a batch of about 32 these layers turn
 * compute-bound): y = x W^T on tcgen05 tensor cores.
 *   x [T][K] (T = B * N tokens), W [Nout][K] (row-major (out, in)), y [T][Nout];
 *   bf16 only (UNSUPPORTED otherwise), fp32 accumulation, y rounded once to
 *   bf16.  K % 8 == 0, pointers 16-byte aligned; y must not overlap x or W
 *   (ALIAS).  The K blocks of all output tiles are divided evenly over the
 *   SMs; a tile whose K range two or more CTAs share is summed from their
 *   fp32 partials in a fixed order (deterministic on a given device); the
 *   scratch for those is medusa_linear_workspace_size(T, K, Nout) bytes (for
 *   the current device; 0 = none needed), 16-byte aligned. */
size_t medusa_linear_workspace_size(int T, int K, int Nout);
medusa_status medusa_linear(const void* x, const void* w, void* y, int T, int K, int Nout, medusa_dtype dt,
                            void* ws, size_t ws_bytes, int32_t* d_status, medusa_stream_t stream);

/* ------------------------------------------------- (h) online tree calibration
 * The sparse tree of the paper review ("方法细节") is built from per-head top-i
 * accuracies measured on calibration data; these calls measure them on the
 * verify steps and rebuild the tree on the device.
 *
 * medusa_accept_stats: adds this step's observations to the counts.  For every
 * batch row, a non-root node n is tested when its parent is on the accepted
 * path and accepted when n is on it (reading: kept on the path; at
 * temperature 0 exactly the argmax-matching child is kept).
 *   path_nodes [B][Dmax+1], accept_len [B] from medusa_typical_accept;
 *   tested, accepted [Dmax][R] uint64, row = depth - 1, column = rank
 *   (caller-owned, zeroed by the caller; atomically incremented).
 *   Dmax >= t->max_depth, t->max_rank <= R <= MEDUSA_MAX_TOPK.
 *   accept_len outside 1..Dmax+1 sets BAD_INDEX (row skipped). */
medusa_status medusa_accept_stats(const int32_t* path_nodes, const int32_t* accept_len,
                                  const medusa_dev_topology* t, int B, int Dmax, int R, uint64_t* tested,
                                  uint64_t* accepted, int32_t* d_status, medusa_stream_t stream);

/* medusa_acc_update: acc[k][i] = (accepted + weight * acc) / (tested + weight)
 * in place on the device table acc [K][R] (fp64), the old table counting as
 * `weight` pseudo-observations; an entry with tested + weight == 0 keeps its
 * value.  Each operation is rounded on its own (IEEE double).  weight >= 0. */
medusa_status medusa_acc_update(double* acc, const uint64_t* tested, const uint64_t* accepted, int K, int R,
                                double weight, medusa_stream_t stream);

/* medusa_topology_greedy_device: the greedy sparse tree of
 * medusa_topology_greedy (same gains, ties and canonical order) built from the
 * device table acc [K][R] (fp64, entries in [0, 1]; others are clamped and set
 * BAD_INDEX) by one CTA, written to the caller's device buffer d_buf
 * (>= medusa_topology_greedy_device_elems(K, n_nodes) int32):
 *   parent[n_nodes], depth[n_nodes], rank[n_nodes], retrieve[n_nodes][K+1].
 * `out` receives pointers into d_buf with n_nodes exact and the bounds
 * max_depth = K, max_rank = R, n_leaves = n_nodes (retrieve rows past the real
 * leaf count are -1); the exact {n_nodes, max_depth, n_leaves, max_rank} are
 * written to d_meta[4].  Enqueued on `stream` like any other call, so later
 * calls on the stream see the new tree.  INVALID_ARG unless
 * 1 + R + ... + R^K >= n_nodes (the tree can always be completed). */
size_t medusa_topology_greedy_device_elems(int K, int n_nodes);
medusa_status medusa_topology_greedy_device(const double* acc, int K, int R, int n_nodes, int32_t* d_buf,
                                            size_t buf_elems, int32_t* d_meta, medusa_dev_topology* out,
                                            int32_t* d_status, medusa_stream_t stream);

/* ------------------------------------------------------------- (i) head loss
 * The Medusa-1 training loss of the K heads and its gradient with respect to
 * the head logits, in one call (paper review, "方法细节": the backbone is
 * frozen and only the heads train, on L1 = -sum_{k=1..K} lambda_k
 * log p_t^(k)(y_{t+k+1}) with lambda_k = 0.8^k; head k read at position t is
 * scored on the token k + 1 places ahead).
 *   logits [K][B][S][V] (`dt`: fp32 or bf16), head k at index k - 1;
 *   tokens [B][S] int32: position t of sequence b counts for head k when
 *   t + k + 1 < S and tokens[b][t+k+1] >= 0 (a negative target is padding and
 *   is skipped); a target >= V sets BAD_INDEX and is skipped.
 *   loss [K + 1] fp32: the mean over the counted positions of -log p of the
 *   target for each head (0 for a head with none), then L1 = sum_k decay^k
 *   times that mean.  Sums run in fp32 in a fixed order (deterministic).
 *   dlogits (`dt`, the layout of logits, or NULL for the loss alone; may be
 *   logits itself, in place, but must not overlap it otherwise):
 *   dL1/dz = decay^k / n_k * (softmax(z) - onehot(target)) on counted rows,
 *   0 on the others (n_k = counted positions of head k).
 *   row_loss [K][B][S] fp32 or NULL: -log p of the target per position (0
 *   where not counted).
 *   1 <= K <= MEDUSA_MAX_HEAD_LOSS_HEADS, K * B * S < 2^31, V >= 1, decay
 *   finite, logits / dlogits aligned to their element size; the scratch is
 *   medusa_head_loss_workspace_size(K, B, S) bytes, 16-byte aligned. */
#define MEDUSA_MAX_HEAD_LOSS_HEADS 32
size_t medusa_head_loss_workspace_size(int K, int B, int S);
medusa_status medusa_head_loss(const void* logits, const int32_t* tokens, int K, int B, int S, int V, float decay,
                               medusa_dtype dt, void* dlogits, float* loss, float* row_loss, void* ws,
                               size_t ws_bytes, int32_t* d_status, medusa_stream_t stream);

/* ------------------------------------------------------------------ status
 * Synchronises `stream`, copies the device status word to *host_code and
 * resets it to 0.  Returns CUDA_ERROR if the stream holds a failed launch. */
medusa_status medusa_status_check(int32_t* d_status, medusa_stream_t stream, int32_t* host_code);

/* Static string naming a medusa_status. */
const char* medusa_status_string(medusa_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int medusa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_GB300_H */
