// Host block manager: reference-counted pool with copy-on-write of a shared
// partial tail, emitting block tables, slots and copy pairs for the kernels.
//
// Behaviour follows "Inside vLLM and TGI: Paging, Versioned Schedulers and
// Operations", section "Exact CPU block manager and copy-on-write" (atomic
// admission, fork by sharing, append with growth or copy-on-write, release
// by reference count, the pool invariants), and the sharing paragraph of
// "vLLM and PagedAttention: Virtual Memory for LLM Serving".  It stores only
// how many positions each block holds, not token contents: the contents live
// in the device pool.  The free-list policy is documented in
// include/pagedkv.h (take from the front, return to the front).
//
// No C++ exception crosses the C ABI: every call that allocates host memory
// does so before it changes any state and returns PKV_ERR_NOMEM if an
// allocation fails, so a failed call leaves the manager as it was.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_block_manager {
  int64_t num_blocks = 0;
  int32_t width = 0;
  std::vector<int32_t> refs;  // tables naming each block
  std::vector<int32_t> fill;  // positions stored in each block
  // The free list as a stack: its back is the front of the list.  Capacity
  // for every block is reserved at creation, so returning a block never
  // allocates.
  std::vector<int32_t> free_list;
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    refs[b] = 1;
    fill[b] = 0;
    return b;
  }
  void unref(int32_t b) {
    if (--refs[b] == 0) {
      fill[b] = 0;
      free_list.push_back(b);
    }
  }
};

namespace {

// The pool invariants that pkv_bm_check reports on (may allocate).
int check_invariants(const pkv_block_manager& m) {
  const pkv_block_manager* bm = &m;
  std::vector<int32_t> count((size_t)bm->num_blocks, 0);
  for (const auto& kv : bm->seqs) {
    const auto& t = kv.second.table;
    if (t.empty()) return PKV_ERR_STATE;
    int64_t held = 0;
    for (size_t j = 0; j < t.size(); ++j) {
      ++count[(size_t)t[j]];
      const int32_t f = bm->fill[(size_t)t[j]];
      if (j + 1 < t.size() ? f != bm->width : (f < 1 || f > bm->width)) return PKV_ERR_STATE;
      held += f;
    }
    if (held != kv.second.len) return PKV_ERR_STATE;
  }
  std::vector<char> in_free((size_t)bm->num_blocks, 0);
  for (int32_t b : bm->free_list) {
    if (in_free[(size_t)b]) return PKV_ERR_STATE;
    in_free[(size_t)b] = 1;
  }
  for (int64_t b = 0; b < bm->num_blocks; ++b) {
    if (bm->refs[(size_t)b] != count[(size_t)b]) return PKV_ERR_STATE;
    if ((bm->refs[(size_t)b] == 0) != (in_free[(size_t)b] != 0)) return PKV_ERR_STATE;
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_block_manager* pkv_bm_create(int64_t num_blocks, int32_t block_size,
                                 const int64_t* free_order) {
  if (num_blocks < 1 || num_blocks > INT32_MAX || block_size < 1) return nullptr;
  auto* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return nullptr;
  try {
    bm->num_blocks = num_blocks;
    bm->width = block_size;
    bm->refs.assign((size_t)num_blocks, 0);
    bm->fill.assign((size_t)num_blocks, 0);
    bm->free_list.reserve((size_t)num_blocks);
    if (free_order) {
      std::vector<char> seen((size_t)num_blocks, 0);
      for (int64_t i = 0; i < num_blocks; ++i) {
        const int64_t b = free_order[i];
        if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
          delete bm;
          return nullptr;
        }
        seen[(size_t)b] = 1;
      }
      for (int64_t i = num_blocks - 1; i >= 0; --i) bm->free_list.push_back((int32_t)free_order[i]);
    } else {
      for (int64_t i = num_blocks - 1; i >= 0; --i) bm->free_list.push_back((int32_t)i);
    }
  } catch (...) {
    delete bm;
    return nullptr;
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_admit(pkv_block_manager* bm, int64_t seq, int64_t num_tokens) {
  if (!bm) return PKV_ERR_NULL;
  if (num_tokens < 1) return PKV_ERR_ARG;
  if (bm->seqs.count(seq)) return PKV_ERR_STATE;
  const int64_t need = num_tokens / bm->width + (num_tokens % bm->width != 0);
  if (need > (int64_t)bm->free_list.size()) return PKV_ERR_NOMEM;
  pkv_block_manager::Seq* s = nullptr;
  try {  // the only allocations, before any block is taken
    pkv_block_manager::Seq fresh;
    fresh.table.reserve((size_t)need);
    s = &bm->seqs.emplace(seq, std::move(fresh)).first->second;
  } catch (...) {
    return PKV_ERR_NOMEM;
  }
  s->len = num_tokens;
  for (int64_t i = 0; i < need; ++i) {
    const int32_t b = bm->take();
    bm->fill[b] = (int32_t)(i + 1 < need ? bm->width : num_tokens - (need - 1) * bm->width);
    s->table.push_back(b);  // within the reserved capacity
  }
  return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return PKV_ERR_NULL;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return PKV_ERR_STATE;
  const std::vector<int32_t>* table = nullptr;
  try {
    pkv_block_manager::Seq copy = it->second;
    table = &bm->seqs.emplace(child, std::move(copy)).first->second.table;
  } catch (...) {
    return PKV_ERR_NOMEM;
  }
  for (int32_t b : *table) ++bm->refs[b];
  return PKV_OK;
}

int pkv_bm_append(pkv_block_manager* bm, const int64_t* seqs, int64_t n, int64_t* slot_mapping,
                  int64_t* pairs, int64_t* num_pairs) {
  if (!bm) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_ARG;
  if (n > 0 && (!seqs || !slot_mapping || !pairs || !num_pairs)) return PKV_ERR_NULL;
  if (num_pairs) *num_pairs = 0;
  // Dry run: count the fresh blocks the whole step needs, following the
  // same decisions as the real pass (earlier appends in the step can lower a
  // shared block's count or fill a fresh block).  Fresh blocks get negative
  // stand-in ids.  Then reserve table room for every append, so that the
  // real pass allocates nothing and cannot fail halfway.
  struct Tail {
    int32_t block;
    int32_t fill;
  };
  int64_t need = 0;
  try {
    std::unordered_map<int64_t, Tail> tails;
    std::unordered_map<int32_t, int32_t> vrefs;
    std::unordered_map<int64_t, int64_t> appends;
    for (int64_t i = 0; i < n; ++i) {
      auto it = bm->seqs.find(seqs[i]);
      if (it == bm->seqs.end()) return PKV_ERR_STATE;
      auto tt = tails.find(seqs[i]);
      Tail t = tt != tails.end() ? tt->second
                                 : Tail{it->second.table.back(), bm->fill[it->second.table.back()]};
      int32_t r = 1;
      if (t.block >= 0) {
        auto rv = vrefs.find(t.block);
        r = rv != vrefs.end() ? rv->second : bm->refs[t.block];
      }
      if (t.fill == bm->width) {
        ++need;
        t = Tail{(int32_t)-need, 1};
      } else if (r > 1) {
        vrefs[t.block] = r - 1;
        ++need;
        t = Tail{(int32_t)-need, t.fill + 1};
      } else {
        ++t.fill;
      }
      tails[seqs[i]] = t;
      ++appends[seqs[i]];
    }
    if (need > (int64_t)bm->free_list.size()) return PKV_ERR_NOMEM;
    for (const auto& kv : appends) {
      auto& table = bm->seqs.find(kv.first)->second.table;
      table.reserve(table.size() + (size_t)kv.second);
    }
  } catch (...) {
    return PKV_ERR_NOMEM;
  }
  int64_t np = 0;
  for (int64_t i = 0; i < n; ++i) {
    auto& s = bm->seqs.find(seqs[i])->second;
    const int32_t last = s.table.back();
    if (bm->fill[last] == bm->width) {
      s.table.push_back(bm->take());  // within the reserved capacity
    } else if (bm->refs[last] > 1) {
      const int32_t fresh = bm->take();
      bm->fill[fresh] = bm->fill[last];
      bm->unref(last);
      s.table.back() = fresh;
      pairs[2 * np] = last;
      pairs[2 * np + 1] = fresh;
      ++np;
    }
    const int32_t tail = s.table.back();
    slot_mapping[i] = (int64_t)tail * bm->width + bm->fill[tail];
    ++bm->fill[tail];
    ++s.len;
  }
  *num_pairs = np;
  return PKV_OK;
}

int pkv_bm_release(pkv_block_manager* bm, int64_t seq) {
  if (!bm) return PKV_ERR_NULL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ERR_STATE;
  for (int32_t b : it->second.table) bm->unref(b);
  bm->seqs.erase(it);
  return PKV_OK;
}

int pkv_bm_tables(const pkv_block_manager* bm, const int64_t* seqs, int64_t n, int32_t max_blocks,
                  int32_t* tables, int32_t* seq_lens) {
  if (!bm) return PKV_ERR_NULL;
  if (n < 0 || max_blocks < 1) return PKV_ERR_ARG;
  if (n > 0 && (!seqs || !tables || !seq_lens)) return PKV_ERR_NULL;
  for (int64_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PKV_ERR_STATE;
    if ((int64_t)it->second.table.size() > max_blocks) return PKV_ERR_CAPACITY;
    if (it->second.len > INT32_MAX) return PKV_ERR_CAPACITY;
  }
  for (int64_t i = 0; i < n; ++i) {
    const auto& s = bm->seqs.find(seqs[i])->second;
    int32_t* row = tables + i * max_blocks;
    const int32_t k = (int32_t)s.table.size();
    for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < k ? s.table[(size_t)j] : -1;
    seq_lens[i] = (int32_t)s.len;
  }
  return PKV_OK;
}

int pkv_bm_slots(const pkv_block_manager* bm, int64_t seq, int64_t start, int64_t count,
                 int64_t* slot_mapping) {
  if (!bm) return PKV_ERR_NULL;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PKV_ERR_STATE;
  if (start < 0 || count < 0 || start > it->second.len || count > it->second.len - start)
    return PKV_ERR_ARG;
  if (count > 0 && !slot_mapping) return PKV_ERR_NULL;
  const auto& table = it->second.table;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t t = start + i;
    slot_mapping[i] = (int64_t)table[(size_t)(t / bm->width)] * bm->width + t % bm->width;
  }
  return PKV_OK;
}

int64_t pkv_bm_num_free(const pkv_block_manager* bm) {
  return bm ? (int64_t)bm->free_list.size() : -1;
}

int64_t pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

int64_t pkv_bm_num_seq_blocks(const pkv_block_manager* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : (int64_t)it->second.table.size();
}

int32_t pkv_bm_refcount(const pkv_block_manager* bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[(size_t)block];
}

int pkv_bm_check(const pkv_block_manager* bm) {
  if (!bm) return PKV_ERR_NULL;
  try {
    return check_invariants(*bm);
  } catch (...) {
    return PKV_ERR_NOMEM;
  }
}

}  // extern "C"
