// Radix tree of cached token runs and their KV-pool slots (host side).
//
// "Inside SGLang", Step 4 (Grow a prefix tree, then run out of room) and the
// "SGLang" notes (RadixAttention: node contents, match_prefix, insertion,
// eviction): a node holds a run of token ids, the pool slots of those tokens,
// its children keyed by first token and a lock count.  A lookup walks down
// while tokens agree and splits a node where the match ends inside it;
// every node it passes gets a new access time.  Insert walks the same way and
// adds the unmatched rest as a leaf, reporting how many tokens were already
// cached (the caller frees their duplicate slots).  A running request locks
// the last node it matched, which covers its path to the root; a split gives
// the new prefix node the lock count of the node it was cut from.  Eviction
// frees unlocked leaves, least recently used first; a parent that becomes a
// leaf is next in line.
//
// Access times come from a logical clock that advances by one per node
// touched (ancestors first); eviction takes the leaf with the smallest
// (access time, creation number).  Node handles carry a generation so a
// handle of an evicted node is rejected rather than aliasing a reused slot.
#include <stdint.h>

#include <algorithm>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/sgl_attn.h"

namespace {

struct Node {
  std::vector<int32_t> key;    // token ids
  std::vector<int32_t> value;  // pool slots, one per token
  std::unordered_map<int32_t, int32_t> children;  // first token -> node index
  int32_t parent = -1;
  int32_t lock_ref = 0;
  int32_t start = 0;           // position of key[0] in any sequence through the node
  uint64_t last_access = 0;
  uint64_t seq = 0;            // creation number
  uint32_t gen = 0;
  bool alive = false;
};

}  // namespace

struct sgl_radix_tree {
  std::vector<Node> nodes;
  std::vector<int32_t> free_ids;
  uint64_t clock = 0, next_seq = 0;
  int64_t evictable = 0, protected_ = 0;

  sgl_radix_tree() {
    const int32_t r = alloc();
    nodes[r].lock_ref = 1;  // the root is never evicted
  }

  int32_t alloc() {
    int32_t id;
    if (!free_ids.empty()) {
      id = free_ids.back();
      free_ids.pop_back();
    } else {
      id = (int32_t)nodes.size();
      nodes.emplace_back();
    }
    Node& n = nodes[id];
    const uint32_t gen = n.gen + 1;
    n = Node();
    n.gen = gen;
    n.alive = true;
    n.seq = next_seq++;
    return id;
  }

  int64_t handle(int32_t id) const { return ((int64_t)nodes[id].gen << 32) | (uint32_t)id; }

  int32_t resolve(int64_t h) const {
    const int64_t id = h & 0xffffffffLL;
    const uint32_t gen = (uint32_t)((uint64_t)h >> 32);
    if (id < 0 || id >= (int64_t)nodes.size()) return -1;
    const Node& n = nodes[id];
    return (n.alive && n.gen == gen) ? (int32_t)id : -1;
  }

  void touch(int32_t id) { nodes[id].last_access = ++clock; }

  // cut node `c` after its first k tokens; returns the new prefix node
  int32_t split(int32_t c, int32_t k) {
    const int32_t nw = alloc();
    Node& child = nodes[c];
    Node& n = nodes[nw];
    n.key.assign(child.key.begin(), child.key.begin() + k);
    n.value.assign(child.value.begin(), child.value.begin() + k);
    n.parent = child.parent;
    n.lock_ref = child.lock_ref;
    n.start = child.start;
    n.last_access = child.last_access;
    child.key.erase(child.key.begin(), child.key.begin() + k);
    child.value.erase(child.value.begin(), child.value.begin() + k);
    child.start += k;
    child.parent = nw;
    nodes[n.parent].children[n.key[0]] = nw;
    n.children[child.key[0]] = c;
    return nw;
  }

  // follow tokens as far as they match; returns the last node and the matched
  // length, appending the path's slots to `slots` when given
  int32_t walk(const int32_t* tok, int32_t n, int32_t* matched, std::vector<int32_t>* slots) {
    int32_t node = 0, pos = 0;
    touch(node);
    for (;;) {
      if (pos >= n) break;
      auto it = nodes[node].children.find(tok[pos]);
      if (it == nodes[node].children.end()) break;
      int32_t c = it->second;
      int32_t k = 0;
      const int32_t len = (int32_t)nodes[c].key.size();
      while (k < len && pos + k < n && nodes[c].key[k] == tok[pos + k]) ++k;
      if (k < len) c = split(c, k);
      touch(c);
      if (slots) slots->insert(slots->end(), nodes[c].value.begin(), nodes[c].value.end());
      pos += k;
      node = c;
    }
    *matched = pos;
    return node;
  }

  bool evictable_leaf(int32_t id) const {
    const Node& n = nodes[id];
    return id != 0 && n.alive && n.children.empty() && n.lock_ref == 0;
  }
};

using Tree = sgl_radix_tree;

extern "C" {

sgl_radix_tree* sgl_radix_create(void) {
  try {
    return new sgl_radix_tree();
  } catch (...) {
    return nullptr;
  }
}

void sgl_radix_destroy(sgl_radix_tree* t) { delete t; }

int32_t sgl_radix_match_prefix(sgl_radix_tree* t, const int32_t* tokens, int32_t n,
                               int32_t* slots_out, int32_t cap, int64_t* node_out) {
  if (!t || n < 0 || cap < 0 || (n > 0 && !tokens) || (cap > 0 && !slots_out)) return -1;
  std::vector<int32_t> slots;
  int32_t matched = 0;
  const int32_t node = t->walk(tokens, n, &matched, &slots);
  const int32_t w = std::min(cap, matched);
  std::copy(slots.begin(), slots.begin() + w, slots_out);
  if (node_out) *node_out = t->handle(node);
  return matched;
}

int32_t sgl_radix_insert(sgl_radix_tree* t, const int32_t* tokens, const int32_t* slots,
                         int32_t n) {
  if (!t || n < 0 || (n > 0 && (!tokens || !slots))) return -1;
  int32_t matched = 0;
  const int32_t node = t->walk(tokens, n, &matched, nullptr);
  if (matched < n) {
    const int32_t leaf = t->alloc();
    Node& l = t->nodes[leaf];
    l.key.assign(tokens + matched, tokens + n);
    l.value.assign(slots + matched, slots + n);
    l.parent = node;
    l.start = matched;
    t->touch(leaf);
    t->nodes[node].children[tokens[matched]] = leaf;
    t->evictable += n - matched;
  }
  return matched;
}

sgl_status sgl_radix_inc_lock_ref(sgl_radix_tree* t, int64_t node) {
  const int32_t id = t ? t->resolve(node) : -1;
  if (id < 0) return SGL_ERR_INVALID_ARG;
  for (int32_t x = id; x != 0; x = t->nodes[x].parent) {
    Node& n = t->nodes[x];
    if (n.lock_ref == 0) {
      t->evictable -= (int64_t)n.key.size();
      t->protected_ += (int64_t)n.key.size();
    }
    ++n.lock_ref;
  }
  return SGL_OK;
}

sgl_status sgl_radix_dec_lock_ref(sgl_radix_tree* t, int64_t node) {
  const int32_t id = t ? t->resolve(node) : -1;
  if (id < 0) return SGL_ERR_INVALID_ARG;
  for (int32_t x = id; x != 0; x = t->nodes[x].parent)
    if (t->nodes[x].lock_ref < 1) return SGL_ERR_INVALID_ARG;  // unbalanced: change nothing
  for (int32_t x = id; x != 0; x = t->nodes[x].parent) {
    Node& n = t->nodes[x];
    if (n.lock_ref == 1) {
      t->evictable += (int64_t)n.key.size();
      t->protected_ -= (int64_t)n.key.size();
    }
    --n.lock_ref;
  }
  return SGL_OK;
}

int32_t sgl_radix_evict(sgl_radix_tree* t, int32_t num_tokens, int32_t* slots_out, int32_t cap) {
  if (!t || num_tokens < 0 || cap < 0 || (cap > 0 && !slots_out)) return -1;
  using Key = std::pair<std::pair<uint64_t, uint64_t>, int32_t>;  // ((time, seq), id)
  std::priority_queue<Key, std::vector<Key>, std::greater<Key>> heap;
  auto push = [&](int32_t id) {
    if (t->evictable_leaf(id))
      heap.push({{t->nodes[id].last_access, t->nodes[id].seq}, id});
  };
  for (int32_t id = 0; id < (int32_t)t->nodes.size(); ++id) push(id);
  int32_t freed = 0;
  while (freed < num_tokens && !heap.empty()) {
    const int32_t id = heap.top().second;
    heap.pop();
    Node& leaf = t->nodes[id];
    const int32_t len = (int32_t)leaf.value.size();
    if (freed + len > cap) break;  // the caller's buffer cannot take this leaf
    std::copy(leaf.value.begin(), leaf.value.end(), slots_out + freed);
    freed += len;
    t->evictable -= len;
    const int32_t parent = leaf.parent;
    t->nodes[parent].children.erase(leaf.key[0]);
    leaf.alive = false;
    leaf.key.clear();
    leaf.value.clear();
    leaf.children.clear();
    t->free_ids.push_back(id);
    push(parent);
  }
  return freed;
}

int64_t sgl_radix_evictable_tokens(const sgl_radix_tree* t) { return t ? t->evictable : -1; }
int64_t sgl_radix_protected_tokens(const sgl_radix_tree* t) { return t ? t->protected_ : -1; }

int32_t sgl_radix_groups(const sgl_radix_tree* t, const int64_t* nodes, int32_t batch,
                         int32_t* group_start, int32_t* group_len, int32_t* group_depth,
                         int32_t* member_off, int32_t* members, int32_t cap_groups,
                         int32_t cap_members, int32_t* n_members_out) {
  if (!t || batch < 0 || (batch > 0 && !nodes) || !n_members_out) return -1;
  // requests through every node on their paths
  std::unordered_map<int32_t, std::vector<int32_t>> through;
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t id = t->resolve(nodes[r]);
    if (id < 0) return -1;
    for (int32_t x = id; x != 0; x = t->nodes[x].parent) through[x].push_back(r);
  }
  struct G {
    int32_t depth, start, len;
    std::vector<int32_t> ms;
  };
  std::vector<G> gs;
  for (auto& kv : through) {
    if (kv.second.size() < 2) continue;
    int32_t depth = 0;
    for (int32_t p = t->nodes[kv.first].parent; p != 0; p = t->nodes[p].parent) ++depth;
    G g{depth, t->nodes[kv.first].start, (int32_t)t->nodes[kv.first].key.size(), kv.second};
    std::sort(g.ms.begin(), g.ms.end());
    gs.push_back(std::move(g));
  }
  std::sort(gs.begin(), gs.end(), [](const G& a, const G& b) {
    if (a.depth != b.depth) return a.depth < b.depth;
    if (a.start != b.start) return a.start < b.start;
    return a.ms[0] < b.ms[0];
  });
  int32_t nm = 0;
  for (const G& g : gs) nm += (int32_t)g.ms.size();
  *n_members_out = nm;
  const int32_t ng = (int32_t)gs.size();
  if (ng > cap_groups || nm > cap_members || !group_start || !group_len || !group_depth ||
      !member_off || !members)
    return ng;  // sizes only
  int32_t off = 0;
  for (int32_t j = 0; j < ng; ++j) {
    group_start[j] = gs[j].start;
    group_len[j] = gs[j].len;
    group_depth[j] = gs[j].depth;
    member_off[j] = off;
    for (int32_t r : gs[j].ms) members[off++] = r;
  }
  member_off[ng] = off;
  return ng;
}

}  // extern "C"
