// phs_cache.cpp -- host-side bookkeeping that feeds block tables to the
// decode kernels: a refcounted page allocator with copy on write, a radix
// prefix tree over whole pages, and the window-safe match length of hybrid
// (Full + SWA) stacks.
//
// Sources:
//  - "Kimi K3 context caching" page, section 1 (global radix tree): requests
//    are matched against a global prefix tree by longest common prefix; a
//    tree node maps to a set of non-contiguous physical KV blocks; requests
//    that hit the same prefix only increment the reference counts of those
//    blocks in the page table (copy on write), and a request's own new
//    tokens get new blocks.  Section 3 sketches match / insert of such a
//    tree (the listing is garbled; only its structure is followed here, with
//    node splitting implemented, which the sketch leaves out).
//  - "Xiaomi MiMo-V2.5 inference system" page, section 2 (prefix cache tree
//    rebuild): with SWA layers a match is valid only at a "window-safe
//    length", where at least the last W tokens still have valid SWA slots;
//    each node carries the Full segment index and the SWA mapping.  Here
//    the SWA mapping is, per cached page, the id of an SWA segment page (a
//    16-token snapshot of that page's SWA-layer KV, saved from the finished
//    request's ring by phs_swa_ring_save) or -1; a window-safe hit returns
//    the segment pages of its last window, which phs_swa_ring_seed copies
//    into the new request's ring.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include "phs.h"

struct phs_page_allocator {
  std::mutex mu;
  std::vector<int32_t> rc;         // reference count per page
  std::vector<int32_t> free_list;  // pages with count 0 (LIFO)
  // the caller's handle plus one per radix tree using this allocator: the
  // object is freed when the last of them lets go, so a tree may outlive
  // the caller's destroy call
  std::atomic<int> holders{1};
};

namespace {

void release_allocator(phs_page_allocator* a) {
  if (a && a->holders.fetch_sub(1) == 1) delete a;
}

int alloc_locked(phs_page_allocator* a, int32_t n, int32_t* out) {
  if (n < 0) return PHS_EINVAL;
  if (static_cast<size_t>(n) > a->free_list.size()) return PHS_ENOSPACE;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = a->free_list.back();
    a->free_list.pop_back();
    a->rc[p] = 1;
    out[i] = p;
  }
  return PHS_OK;
}

bool valid_page(const phs_page_allocator* a, int32_t p) {
  return p >= 0 && static_cast<size_t>(p) < a->rc.size();
}

int incref_locked(phs_page_allocator* a, const int32_t* pages, int32_t n) {
  for (int32_t i = 0; i < n; ++i)
    if (!valid_page(a, pages[i]) || a->rc[pages[i]] <= 0) return PHS_ERANGE;
  for (int32_t i = 0; i < n; ++i) ++a->rc[pages[i]];
  return PHS_OK;
}

int decref_locked(phs_page_allocator* a, const int32_t* pages, int32_t n) {
  for (int32_t i = 0; i < n; ++i)
    if (!valid_page(a, pages[i]) || a->rc[pages[i]] <= 0) return PHS_ERANGE;
  for (int32_t i = 0; i < n; ++i)
    if (--a->rc[pages[i]] == 0) a->free_list.push_back(pages[i]);
  return PHS_OK;
}

}  // namespace

extern "C" {

phs_page_allocator* phs_page_allocator_create(int64_t num_pages) {
  if (num_pages <= 0 || num_pages > INT32_MAX) return nullptr;
  auto* a = new phs_page_allocator();
  a->rc.assign(static_cast<size_t>(num_pages), 0);
  a->free_list.reserve(static_cast<size_t>(num_pages));
  for (int64_t p = num_pages - 1; p >= 0; --p) a->free_list.push_back(static_cast<int32_t>(p));
  return a;
}

void phs_page_allocator_destroy(phs_page_allocator* a) { release_allocator(a); }

int phs_page_alloc(phs_page_allocator* a, int32_t n, int32_t* out_pages) {
  if (!a || (n > 0 && !out_pages)) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  return alloc_locked(a, n, out_pages);
}

int phs_page_incref(phs_page_allocator* a, const int32_t* pages, int32_t n) {
  if (!a || n < 0 || (n > 0 && !pages)) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  return incref_locked(a, pages, n);
}

int phs_page_decref(phs_page_allocator* a, const int32_t* pages, int32_t n) {
  if (!a || n < 0 || (n > 0 && !pages)) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  return decref_locked(a, pages, n);
}

int64_t phs_page_free_count(phs_page_allocator* a) {
  if (!a) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  return static_cast<int64_t>(a->free_list.size());
}

int phs_page_refcounts(phs_page_allocator* a, int32_t* out) {
  if (!a || !out) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  std::memcpy(out, a->rc.data(), a->rc.size() * sizeof(int32_t));
  return PHS_OK;
}

int phs_page_cow(phs_page_allocator* a, int32_t page, int32_t* out_page) {
  if (!a || !out_page) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(a->mu);
  if (!valid_page(a, page) || a->rc[page] <= 0) return PHS_ERANGE;
  if (a->rc[page] == 1) {
    *out_page = page;
    return PHS_OK;
  }
  int32_t fresh;
  const int st = alloc_locked(a, 1, &fresh);
  if (st) return st;
  --a->rc[page];  // > 0 remains: still shared by the others
  *out_page = fresh;
  return PHS_OK;
}

int64_t phs_window_safe_len(const uint8_t* swa_valid, int64_t match_len, int32_t window,
                            int32_t align) {
  if (match_len < 0 || window <= 0 || align <= 0 || (match_len > 0 && !swa_valid))
    return PHS_EINVAL;
  // run = number of consecutive valid positions ending at t (exclusive end)
  int64_t best = 0, run = 0;
  for (int64_t L = 1; L <= match_len; ++L) {
    run = swa_valid[L - 1] ? run + 1 : 0;
    const int64_t need = L < window ? L : window;
    if (L % align == 0 && run >= need) best = L;
  }
  return best;
}

}  // extern "C"

// ----------------------------------------------------------------- radix --
namespace {

struct Node {
  std::vector<int32_t> tokens;  // a whole number of pages' tokens
  std::vector<int32_t> pages;   // tokens.size() / page_size page ids
  std::vector<int32_t> swa;     // per page: SWA segment page id, or -1
  // by the tokens of the child's first page (sharing is by whole pages)
  std::map<std::vector<int32_t>, std::unique_ptr<Node>> children;
  Node* parent = nullptr;
  uint64_t last_access = 0;
};

}  // namespace

struct phs_radix_tree {
  std::mutex mu;
  phs_page_allocator* alloc = nullptr;
  phs_page_allocator* swa_alloc = nullptr;  // SWA segment pages (may be null)
  int32_t P = 16;
  Node root;
  uint64_t clock = 0;
  int64_t cached_pages = 0;
};

namespace {

// whole pages of node `c` that match tokens[idx..n)
int64_t pages_matching(const phs_radix_tree* t, const Node* c, const int32_t* tokens, int64_t idx,
                       int64_t n) {
  const int64_t P = t->P;
  int64_t k = 0;
  const int64_t np = static_cast<int64_t>(c->pages.size());
  while (k < np && idx + (k + 1) * P <= n &&
         std::equal(c->tokens.begin() + k * P, c->tokens.begin() + (k + 1) * P,
                    tokens + idx + k * P))
    ++k;
  return k;
}

// Split node c after k pages: c keeps the first k pages, a new child holds
// the rest (and inherits c's children).
void split(phs_radix_tree* t, Node* c, int64_t k) {
  const int64_t P = t->P;
  auto tail = std::make_unique<Node>();
  tail->tokens.assign(c->tokens.begin() + k * P, c->tokens.end());
  tail->pages.assign(c->pages.begin() + k, c->pages.end());
  tail->swa.assign(c->swa.begin() + k, c->swa.end());
  tail->children = std::move(c->children);
  for (auto& kv : tail->children) kv.second->parent = tail.get();
  tail->parent = c;
  tail->last_access = c->last_access;
  c->tokens.resize(k * P);
  c->pages.resize(k);
  c->swa.resize(k);
  c->children.clear();
  std::vector<int32_t> key(tail->tokens.begin(), tail->tokens.begin() + P);
  c->children[std::move(key)] = std::move(tail);
}

// Walk the longest whole-page match; appends pages and their SWA segment ids.
void walk_match(phs_radix_tree* t, const int32_t* tokens, int64_t n, std::vector<int32_t>& pages,
                std::vector<int32_t>& swa) {
  Node* cur = &t->root;
  int64_t idx = 0;
  const uint64_t now = ++t->clock;
  while (idx + t->P <= n) {
    auto it = cur->children.find(std::vector<int32_t>(tokens + idx, tokens + idx + t->P));
    if (it == cur->children.end()) break;
    Node* c = it->second.get();
    const int64_t k = pages_matching(t, c, tokens, idx, n);
    if (k == 0) break;
    pages.insert(pages.end(), c->pages.begin(), c->pages.begin() + k);
    swa.insert(swa.end(), c->swa.begin(), c->swa.begin() + k);
    for (Node* u = c; u; u = u->parent) u->last_access = now;
    idx += k * t->P;
    if (k < static_cast<int64_t>(c->pages.size())) break;
    cur = c;
  }
}

int finish_match(phs_radix_tree* t, std::vector<int32_t>& pages, int64_t keep_pages,
                 int32_t* out_pages, int32_t max_pages, int32_t* out_num_pages) {
  pages.resize(static_cast<size_t>(keep_pages));
  if (keep_pages > max_pages) return PHS_ESHAPE;
  {
    std::lock_guard<std::mutex> lock(t->alloc->mu);
    const int st = incref_locked(t->alloc, pages.data(), static_cast<int32_t>(keep_pages));
    if (st) return st;
  }
  std::copy(pages.begin(), pages.end(), out_pages);
  *out_num_pages = static_cast<int32_t>(keep_pages);
  return PHS_OK;
}

// Drop the tree's references on the SWA segment pages of a node (ids >= 0).
void release_swa_locked(phs_radix_tree* t, const std::vector<int32_t>& swa) {
  if (!t->swa_alloc) return;
  std::vector<int32_t> held;
  for (int32_t s : swa)
    if (s >= 0) held.push_back(s);
  decref_locked(t->swa_alloc, held.data(), static_cast<int32_t>(held.size()));
}

void collect_leaves(Node* n, std::vector<Node*>& out) {
  for (auto& kv : n->children) {
    if (kv.second->children.empty())
      out.push_back(kv.second.get());
    else
      collect_leaves(kv.second.get(), out);
  }
}

}  // namespace

extern "C" {

phs_radix_tree* phs_radix_create(phs_page_allocator* alloc, phs_page_allocator* swa_alloc,
                                 int32_t page_size) {
  if (!alloc || page_size <= 0 || swa_alloc == alloc) return nullptr;
  auto* t = new phs_radix_tree();
  t->alloc = alloc;
  t->swa_alloc = swa_alloc;
  t->P = page_size;
  alloc->holders.fetch_add(1);
  if (swa_alloc) swa_alloc->holders.fetch_add(1);
  return t;
}

void phs_radix_destroy(phs_radix_tree* t) {
  if (!t) return;
  // drop the tree's reference on every cached page
  std::vector<Node*> stack;
  for (auto& kv : t->root.children) stack.push_back(kv.second.get());
  {
    std::lock_guard<std::mutex> lock(t->alloc->mu);
    std::unique_lock<std::mutex> slock;
    if (t->swa_alloc) slock = std::unique_lock<std::mutex>(t->swa_alloc->mu);
    while (!stack.empty()) {
      Node* n = stack.back();
      stack.pop_back();
      decref_locked(t->alloc, n->pages.data(), static_cast<int32_t>(n->pages.size()));
      release_swa_locked(t, n->swa);
      for (auto& kv : n->children) stack.push_back(kv.second.get());
    }
  }
  release_allocator(t->alloc);
  release_allocator(t->swa_alloc);
  delete t;
}

int phs_radix_match(phs_radix_tree* t, const int32_t* tokens, int64_t n, int32_t* out_pages,
                    int32_t max_pages, int32_t* out_num_pages) {
  if (!t || n < 0 || (n > 0 && !tokens) || !out_num_pages || (max_pages > 0 && !out_pages))
    return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(t->mu);
  std::vector<int32_t> pages;
  std::vector<int32_t> swa;
  walk_match(t, tokens, n, pages, swa);
  return finish_match(t, pages, static_cast<int64_t>(pages.size()), out_pages, max_pages,
                      out_num_pages);
}

int phs_radix_match_window_safe(phs_radix_tree* t, const int32_t* tokens, int64_t n,
                                int32_t window, int32_t* out_pages, int32_t max_pages,
                                int32_t* out_num_pages, int32_t* out_swa_pages,
                                int32_t max_swa_pages, int32_t* out_num_swa_pages) {
  if (!t || n < 0 || window <= 0 || (n > 0 && !tokens) || !out_num_pages ||
      (max_pages > 0 && !out_pages) || !out_num_swa_pages ||
      (max_swa_pages > 0 && !out_swa_pages))
    return PHS_EINVAL;
  if (window % t->P != 0) return PHS_EUNSUPPORTED;  // the window is whole pages
  std::lock_guard<std::mutex> lock(t->mu);
  std::vector<int32_t> pages;
  std::vector<int32_t> swa;
  walk_match(t, tokens, n, pages, swa);
  // per-token validity: a token has SWA KV where its page has a segment page
  std::vector<uint8_t> valid(pages.size() * static_cast<size_t>(t->P));
  for (size_t i = 0; i < valid.size(); ++i) valid[i] = swa[i / t->P] >= 0 ? 1 : 0;
  const int64_t L = phs_window_safe_len(valid.data(), static_cast<int64_t>(valid.size()),
                                        window, t->P);
  if (L < 0) return static_cast<int>(L);
  const int64_t keep = L / t->P;
  const int64_t first = (L - std::min<int64_t>(L, window)) / t->P;  // the last window's pages
  const int64_t nswa = keep - first;
  if (nswa > max_swa_pages) return PHS_ESHAPE;
  if (nswa > 0 && !t->swa_alloc) return PHS_EINVAL;
  std::vector<int32_t> seg(swa.begin() + first, swa.begin() + keep);
  if (nswa > 0) {
    std::lock_guard<std::mutex> slock(t->swa_alloc->mu);
    const int st = incref_locked(t->swa_alloc, seg.data(), static_cast<int32_t>(nswa));
    if (st) return st;
  }
  const int st = finish_match(t, pages, keep, out_pages, max_pages, out_num_pages);
  if (st) {
    if (nswa > 0) {
      std::lock_guard<std::mutex> slock(t->swa_alloc->mu);
      decref_locked(t->swa_alloc, seg.data(), static_cast<int32_t>(nswa));
    }
    return st;
  }
  std::copy(seg.begin(), seg.end(), out_swa_pages);
  *out_num_swa_pages = static_cast<int32_t>(nswa);
  return PHS_OK;
}

int phs_radix_insert(phs_radix_tree* t, const int32_t* tokens, int64_t n, const int32_t* pages,
                     const int32_t* swa_pages) {
  if (!t || n < 0 || (n > 0 && (!tokens || !pages))) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(t->mu);
  const int64_t P = t->P;
  const int64_t np = n / P;  // only whole pages are shared
  const uint64_t now = ++t->clock;
  auto swa_of = [&](int64_t page) { return swa_pages ? swa_pages[page] : -1; };
  if (swa_pages) {
    bool any = false;
    for (int64_t i = 0; i < np; ++i) any = any || swa_pages[i] >= 0;
    if (any && !t->swa_alloc) return PHS_EINVAL;
  }
  Node* cur = &t->root;
  int64_t idx = 0;  // tokens consumed
  while (idx < np * P) {
    auto it = cur->children.find(std::vector<int32_t>(tokens + idx, tokens + idx + P));
    if (it != cur->children.end()) {
      Node* c = it->second.get();
      const int64_t k = pages_matching(t, c, tokens, idx, np * P);
      if (k > 0) {
        if (k < static_cast<int64_t>(c->pages.size())) split(t, c, k);
        // a cached page without SWA KV takes the caller's segment page (the
        // tree takes a reference on it); one that has one keeps it
        for (int64_t i = 0; i < k; ++i) {
          const int32_t s = swa_of(idx / P + i);
          if (c->swa[i] < 0 && s >= 0) {
            std::lock_guard<std::mutex> slock(t->swa_alloc->mu);
            const int st = incref_locked(t->swa_alloc, &s, 1);
            if (st) return st;
            c->swa[i] = s;
          }
        }
        c->last_access = now;
        idx += k * P;
        cur = c;
        continue;
      }
    }
    // new leaf with the remaining whole pages; the tree takes a reference
    auto leaf = std::make_unique<Node>();
    leaf->tokens.assign(tokens + idx, tokens + np * P);
    leaf->pages.assign(pages + idx / P, pages + np);
    leaf->swa.resize(leaf->pages.size());
    for (size_t i = 0; i < leaf->swa.size(); ++i) leaf->swa[i] = swa_of(idx / P + i);
    leaf->parent = cur;
    leaf->last_access = now;
    {
      std::lock_guard<std::mutex> alock(t->alloc->mu);
      int st = incref_locked(t->alloc, leaf->pages.data(),
                             static_cast<int32_t>(leaf->pages.size()));
      if (st) return st;
      if (t->swa_alloc) {
        std::vector<int32_t> held;
        for (int32_t s : leaf->swa)
          if (s >= 0) held.push_back(s);
        std::lock_guard<std::mutex> slock(t->swa_alloc->mu);
        st = incref_locked(t->swa_alloc, held.data(), static_cast<int32_t>(held.size()));
        if (st) {
          decref_locked(t->alloc, leaf->pages.data(), static_cast<int32_t>(leaf->pages.size()));
          return st;
        }
      }
    }
    t->cached_pages += static_cast<int64_t>(leaf->pages.size());
    std::vector<int32_t> key(leaf->tokens.begin(), leaf->tokens.begin() + P);
    cur->children[std::move(key)] = std::move(leaf);
    break;
  }
  return PHS_OK;
}

int phs_radix_evict(phs_radix_tree* t, int64_t pages, int64_t* out_freed) {
  if (!t || pages < 0 || !out_freed) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(t->mu);
  int64_t freed = 0;
  while (freed < pages) {
    std::vector<Node*> leaves;
    collect_leaves(&t->root, leaves);
    std::sort(leaves.begin(), leaves.end(),
              [](const Node* a, const Node* b) { return a->last_access < b->last_access; });
    Node* victim = nullptr;
    {
      std::lock_guard<std::mutex> alock(t->alloc->mu);
      std::unique_lock<std::mutex> slock;
      if (t->swa_alloc) slock = std::unique_lock<std::mutex>(t->swa_alloc->mu);
      for (Node* l : leaves) {
        bool only_tree = true;
        for (int32_t p : l->pages) only_tree = only_tree && t->alloc->rc[p] == 1;
        if (t->swa_alloc)
          for (int32_t s : l->swa) only_tree = only_tree && (s < 0 || t->swa_alloc->rc[s] == 1);
        if (only_tree) {
          victim = l;
          break;
        }
      }
      if (!victim) break;  // every cached leaf is in use by some request
      decref_locked(t->alloc, victim->pages.data(), static_cast<int32_t>(victim->pages.size()));
      release_swa_locked(t, victim->swa);
    }
    freed += static_cast<int64_t>(victim->pages.size());
    t->cached_pages -= static_cast<int64_t>(victim->pages.size());
    Node* parent = victim->parent;
    parent->children.erase(
        std::vector<int32_t>(victim->tokens.begin(), victim->tokens.begin() + t->P));
  }
  *out_freed = freed;
  return PHS_OK;
}

int64_t phs_radix_cached_pages(phs_radix_tree* t) {
  if (!t) return PHS_EINVAL;
  std::lock_guard<std::mutex> lock(t->mu);
  return t->cached_pages;
}

}  // extern "C"
