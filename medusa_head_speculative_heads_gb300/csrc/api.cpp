// Host side of libmedusa_gb300: candidate-tree topology builders, topology
// upload, device status word, version.
//
// Topology (skill-pack guide "Medusa 多解码头推理加速全解析", sections "候选生成"
// and "树结构：medusa_choices"; paper review "Medusa: Simple LLM Inference
// Acceleration Framework with Multiple Decoding Heads", section "方法细节",
// sparse tree construction).  A node is its rank path (element j = rank within
// Medusa head j+1's top-k).  Canonical order sorts paths by (length,
// lexicographic), so the root is node 0 and parents precede children.
#include <atomic>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <set>
#include <vector>

#include "host_util.h"
#include "medusa.h"

namespace medusa {

using Path = std::vector<int32_t>;

static bool canonical_less(const Path& a, const Path& b) {
  if (a.size() != b.size()) return a.size() < b.size();
  return a < b;
}

// Fills `out` from a canonical, ancestor-closed path list (paths[0] empty).
static medusa_status fill_topology(const std::vector<Path>& paths, medusa_topology* out) {
  const int n = (int)paths.size();
  if (n < 1 || n > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  std::map<Path, int> index;
  for (int i = 0; i < n; ++i) index[paths[i]] = i;
  out->n_nodes = n;
  int max_depth = 0, max_rank = 0;
  std::vector<char> has_child(n, 0);
  for (int i = 0; i < n; ++i) {
    const Path& p = paths[i];
    if ((int)p.size() > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
    out->depth[i] = (int32_t)p.size();
    if (i == 0) {
      out->parent[i] = -1;
      out->rank[i] = -1;
      continue;
    }
    Path par(p.begin(), p.end() - 1);
    auto it = index.find(par);
    if (it == index.end() || it->second >= i) return MEDUSA_ERR_INVALID_ARG;
    out->parent[i] = it->second;
    out->rank[i] = p.back();
    has_child[it->second] = 1;
    max_depth = std::max(max_depth, (int)p.size());
    max_rank = std::max(max_rank, p.back() + 1);
  }
  out->max_depth = max_depth;
  out->max_rank = max_rank;
  int leaves = 0;
  for (int i = 0; i < n; ++i) {
    if (has_child[i]) continue;
    int32_t* row = out->retrieve + (size_t)leaves * (max_depth + 1);
    for (int j = 0; j <= max_depth; ++j) row[j] = -1;
    for (int a = i; a >= 0; a = out->parent[a]) row[out->depth[a]] = a;
    ++leaves;
  }
  out->n_leaves = leaves;
  return MEDUSA_OK;
}

// Per-device cache; concurrent first calls may both query, and store the same value.
static std::atomic<int> cached_sm_count[64];

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kNumSMsFallback;
  int n = cached_sm_count[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kNumSMsFallback;
    cached_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace medusa

using namespace medusa;

extern "C" medusa_status medusa_topology_from_paths(const int32_t* ranks, const int32_t* path_len,
                                                    int n_paths, int max_nodes,
                                                    medusa_topology* out) {
  if (!out || n_paths < 0 || (n_paths > 0 && (!ranks || !path_len))) return MEDUSA_ERR_INVALID_ARG;
  if (max_nodes < 1 || max_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  std::set<Path> s;
  s.insert(Path());
  size_t off = 0;
  for (int i = 0; i < n_paths; ++i) {
    const int len = path_len[i];
    if (len < 1 || len > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
    Path p(ranks + off, ranks + off + len);
    off += (size_t)len;
    for (int32_t r : p)
      if (r < 0 || r >= MEDUSA_MAX_TOPK) return MEDUSA_ERR_INVALID_ARG;
    s.insert(p);
  }
  for (const Path& p : s)
    if (!p.empty() && !s.count(Path(p.begin(), p.end() - 1))) return MEDUSA_ERR_INVALID_ARG;
  if ((int)s.size() > max_nodes) return MEDUSA_ERR_INVALID_ARG;
  std::vector<Path> v(s.begin(), s.end());
  std::sort(v.begin(), v.end(), canonical_less);
  return fill_topology(v, out);
}

extern "C" medusa_status medusa_topology_dense(int K, const int32_t* topk_per_head, int max_nodes,
                                               medusa_topology* out) {
  if (!out || !topk_per_head || K < 1 || K > MEDUSA_MAX_DEPTH) return MEDUSA_ERR_INVALID_ARG;
  if (max_nodes < 1 || max_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  for (int j = 0; j < K; ++j)
    if (topk_per_head[j] < 1 || topk_per_head[j] > MEDUSA_MAX_TOPK) return MEDUSA_ERR_INVALID_ARG;
  // Level by level in canonical order; each level is the lexicographic
  // enumeration of rank tuples, so stop as soon as the budget is reached.
  std::vector<Path> v;
  v.push_back(Path());
  std::vector<Path> level(1, Path());
  for (int depth = 1; depth <= K && (int)v.size() < max_nodes; ++depth) {
    std::vector<Path> next;
    for (const Path& p : level)
      for (int r = 0; r < topk_per_head[depth - 1]; ++r) {
        Path c = p;
        c.push_back(r);
        next.push_back(c);
      }
    for (const Path& c : next) {
      if ((int)v.size() >= max_nodes) break;
      v.push_back(c);
    }
    level.swap(next);
  }
  return fill_topology(v, out);
}

extern "C" medusa_status medusa_topology_greedy(const double* acc, int K, int R, int n_nodes,
                                                medusa_topology* out) {
  if (!out || !acc || K < 1 || K > MEDUSA_MAX_DEPTH || R < 1 || R > MEDUSA_MAX_TOPK)
    return MEDUSA_ERR_INVALID_ARG;
  if (n_nodes < 1 || n_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  for (int i = 0; i < K * R; ++i)
    if (!(acc[i] >= 0.0) || !(acc[i] <= 1.0)) return MEDUSA_ERR_INVALID_ARG;
  // Chosen nodes with their reach probability; the frontier is every child
  // (one more head, any rank) of a chosen node that is not chosen yet.
  std::vector<Path> chosen(1, Path());
  std::vector<double> chosen_score(1, 1.0);
  std::set<Path> in_tree;
  in_tree.insert(Path());
  while ((int)chosen.size() < n_nodes) {
    bool found = false;
    double best_s = 0.0;
    Path best_p;
    for (size_t a = 0; a < chosen.size(); ++a) {
      const Path& p = chosen[a];
      if ((int)p.size() >= K) continue;
      const int head = (int)p.size();
      for (int r = 0; r < R; ++r) {
        Path c = p;
        c.push_back(r);
        if (in_tree.count(c)) continue;
        const double sc = chosen_score[a] * acc[head * R + r];
        bool better;
        if (!found) {
          better = true;
        } else if (std::fabs(sc - best_s) <= 1e-12 * std::max(std::fabs(sc), std::fabs(best_s))) {
          better = canonical_less(c, best_p);
        } else {
          better = sc > best_s;
        }
        if (better) {
          found = true;
          best_s = sc;
          best_p = c;
        }
      }
    }
    if (!found) break;
    chosen.push_back(best_p);
    chosen_score.push_back(best_s);
    in_tree.insert(best_p);
  }
  std::sort(chosen.begin(), chosen.end(), canonical_less);
  return fill_topology(chosen, out);
}

extern "C" size_t medusa_topology_device_elems(const medusa_topology* t) {
  if (!t || t->n_nodes < 1) return 0;
  return (size_t)3 * t->n_nodes + (size_t)t->n_leaves * (t->max_depth + 1);
}

extern "C" medusa_status medusa_topology_upload(const medusa_topology* t, int32_t* d_buf,
                                                size_t buf_elems, medusa_dev_topology* out,
                                                medusa_stream_t stream) {
  if (!t || !d_buf || !out || t->n_nodes < 1 || t->n_nodes > MEDUSA_MAX_NODES) return MEDUSA_ERR_INVALID_ARG;
  const size_t need = medusa_topology_device_elems(t);
  if (buf_elems < need) return MEDUSA_ERR_INVALID_ARG;
  const int n = t->n_nodes;
  std::vector<int32_t> host(need);
  std::memcpy(host.data(), t->parent, sizeof(int32_t) * n);
  std::memcpy(host.data() + n, t->depth, sizeof(int32_t) * n);
  std::memcpy(host.data() + 2 * n, t->rank, sizeof(int32_t) * n);
  std::memcpy(host.data() + 3 * n, t->retrieve, sizeof(int32_t) * t->n_leaves * (t->max_depth + 1));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(d_buf, host.data(), need * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MEDUSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEDUSA_ERR_CUDA;
  out->n_nodes = n;
  out->max_depth = t->max_depth;
  out->n_leaves = t->n_leaves;
  out->max_rank = t->max_rank;
  out->parent = d_buf;
  out->depth = d_buf + n;
  out->rank = d_buf + 2 * n;
  out->retrieve = d_buf + 3 * n;
  return MEDUSA_OK;
}

extern "C" medusa_status medusa_status_check(int32_t* d_status, medusa_stream_t stream,
                                             int32_t* host_code) {
  if (!d_status || !host_code) return MEDUSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, d_status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaMemsetAsync(d_status, 0, sizeof v, s) != cudaSuccess) return MEDUSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MEDUSA_ERR_CUDA;
  *host_code = v;
  return MEDUSA_OK;
}

extern "C" const char* medusa_status_string(medusa_status s) {
  switch (s) {
    case MEDUSA_OK: return "MEDUSA_OK";
    case MEDUSA_ERR_INVALID_ARG: return "MEDUSA_ERR_INVALID_ARG";
    case MEDUSA_ERR_UNSUPPORTED: return "MEDUSA_ERR_UNSUPPORTED";
    case MEDUSA_ERR_ALIAS: return "MEDUSA_ERR_ALIAS";
    case MEDUSA_ERR_CUDA: return "MEDUSA_ERR_CUDA";
    case MEDUSA_ERR_WORKSPACE: return "MEDUSA_ERR_WORKSPACE";
  }
  return "MEDUSA_ERR_UNKNOWN";
}

extern "C" int medusa_version(void) { return 100; }
