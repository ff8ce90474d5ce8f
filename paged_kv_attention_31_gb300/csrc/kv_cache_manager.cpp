// kv_cache_manager.cpp -- host-side page manager of the paged KV pool: hands
// pool blocks to sequences, shares prefix blocks between sequences, copies a
// shared block before a sequence writes into it, and preempts sequences last
// in, first out when the pool runs short.  Its outputs are exactly the inputs
// of the device calls: slot mappings for pkv_kv_append, (source, destination)
// block pairs for pkv_copy_blocks, and block tables / context lengths for
// pkv_paged_attention and pkv_paged_prefill.
//
// "TensorRT-LLM框架解析与高性能推理优化实践" §4.1 (the KV-cache manager:
// paged cache, block reuse and prefix sharing, reclaiming memory) and §4.2
// (KV缓存管理细节: blocks of one pool, allocate / free, a block list per
// sequence); §5.2 (抢占策略实现: the most recently admitted running request is
// preempted first, its blocks freed, until the new request fits).
//
// Policy (fixed so that results are reproducible id for id):
//   * free blocks form a stack; block 0 starts on top; allocation pops,
//     release pushes;
//   * fork(parent, child, n) shares the parent's first ceil(n / P) blocks;
//   * a block with more than one owner is copied before a sequence writes into
//     it: a fresh block is popped and the pair (old, new) is reported;
//   * append is all-or-nothing over all its sequences;
//   * release pushes a sequence's blocks last page first; a block is free when
//     its owner count reaches zero;
//   * preempt_for frees whole sequences in reverse admission order, skipping
//     protected ones, and changes nothing if that cannot free enough.
//
// All work is O(blocks touched): the free stack and the owner counts are flat
// arrays, sequences are found by hash, admission order is an ordered map.
#include <cstdint>
#include <map>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pkv.h"

struct pkv_cache {
  struct Seq {
    std::vector<int32_t> pages;
    int32_t len = 0;
    int64_t admitted = 0;
  };
  int32_t num_blocks = 0, block_size = 0, max_blocks = 0;
  std::vector<int32_t> free_stack;            // top = back()
  std::vector<int32_t> owners;                // per block
  std::unordered_map<int64_t, Seq> seqs;
  std::map<int64_t, int64_t> by_admission;    // admission number -> seq id
  int64_t admitted = 0;
  // scratch for all-or-nothing planning: owner-count deltas of touched blocks
  std::vector<int32_t> delta;
  std::vector<int32_t> touched;

  void reset_delta() {
    for (int32_t b : touched) delta[b] = 0;
    touched.clear();
  }
  void add_delta(int32_t b, int32_t d) {
    if (delta[b] == 0) touched.push_back(b);
    delta[b] += d;
  }
  int32_t pop_block() {
    const int32_t b = free_stack.back();
    free_stack.pop_back();
    owners[b] = 1;
    return b;
  }
  void drop_block(int32_t b) {
    if (--owners[b] == 0) free_stack.push_back(b);
  }

  // Blocks that appending counts[i] tokens to seq_ids[i] needs (new pages plus
  // copies), or -1 if the request is invalid.
  int64_t plan(const int64_t* ids, const int32_t* counts, int32_t n) {
    int64_t need = 0;
    std::unordered_set<int64_t> seen;
    seen.reserve(size_t(n) * 2);
    bool ok = true;
    for (int32_t i = 0; i < n && ok; ++i) {
      auto it = seqs.find(ids[i]);
      if (it == seqs.end() || counts[i] < 0 || !seen.insert(ids[i]).second) {
        ok = false;
        break;
      }
      const Seq& s = it->second;
      const int64_t end = int64_t(s.len) + counts[i];
      if ((end + block_size - 1) / block_size > max_blocks) {
        ok = false;
        break;
      }
      if (counts[i] == 0) continue;
      const int64_t first = s.len / block_size, last = (end - 1) / block_size;
      for (int64_t j = first; j <= last; ++j) {
        if (j < int64_t(s.pages.size())) {
          const int32_t b = s.pages[size_t(j)];
          if (owners[b] + delta[b] > 1) {   // shared: one copy, one owner less
            add_delta(b, -1);
            ++need;
          }
        } else {
          ++need;
        }
      }
    }
    reset_delta();
    return ok ? need : -1;
  }
};

extern "C" {

pkv_status pkv_cache_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                            pkv_cache** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
  if (int64_t(num_blocks) * block_size > (int64_t(1) << 62)) return PKV_ERR_INVALID_ARG;
  pkv_cache* c = new (std::nothrow) pkv_cache;
  if (!c) return PKV_ERR_INVALID_ARG;
  try {
    c->num_blocks = num_blocks;
    c->block_size = block_size;
    c->max_blocks = max_blocks_per_seq;
    c->free_stack.resize(size_t(num_blocks));
    for (int32_t i = 0; i < num_blocks; ++i) c->free_stack[size_t(i)] = num_blocks - 1 - i;
    c->owners.assign(size_t(num_blocks), 0);
    c->delta.assign(size_t(num_blocks), 0);
  } catch (...) {
    delete c;
    return PKV_ERR_INVALID_ARG;
  }
  *out = c;
  return PKV_OK;
}

void pkv_cache_destroy(pkv_cache* c) { delete c; }

int32_t pkv_cache_num_free(const pkv_cache* c) {
  return c ? int32_t(c->free_stack.size()) : -1;
}

int32_t pkv_cache_num_seqs(const pkv_cache* c) { return c ? int32_t(c->seqs.size()) : -1; }

int32_t pkv_cache_length(const pkv_cache* c, int64_t seq_id) {
  if (!c) return -1;
  auto it = c->seqs.find(seq_id);
  return it == c->seqs.end() ? -1 : it->second.len;
}

pkv_status pkv_cache_add(pkv_cache* c, int64_t seq_id) {
  if (!c || seq_id < 0 || c->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  pkv_cache::Seq s;
  s.admitted = c->admitted++;
  c->by_admission.emplace(s.admitted, seq_id);
  c->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

pkv_status pkv_cache_fork(pkv_cache* c, int64_t parent, int64_t child, int32_t num_tokens) {
  if (!c || child < 0 || c->seqs.count(child)) return PKV_ERR_INVALID_ARG;
  auto it = c->seqs.find(parent);
  if (it == c->seqs.end() || num_tokens < 0 || num_tokens > it->second.len)
    return PKV_ERR_INVALID_ARG;
  pkv_cache::Seq s;
  const size_t n = size_t((int64_t(num_tokens) + c->block_size - 1) / c->block_size);
  s.pages.assign(it->second.pages.begin(), it->second.pages.begin() + long(n));
  for (int32_t b : s.pages) ++c->owners[b];
  s.len = num_tokens;
  s.admitted = c->admitted++;
  c->by_admission.emplace(s.admitted, child);
  c->seqs.emplace(child, std::move(s));
  return PKV_OK;
}

pkv_status pkv_cache_release(pkv_cache* c, int64_t seq_id) {
  if (!c) return PKV_ERR_INVALID_ARG;
  auto it = c->seqs.find(seq_id);
  if (it == c->seqs.end()) return PKV_ERR_INVALID_ARG;
  const auto& pages = it->second.pages;
  for (auto b = pages.rbegin(); b != pages.rend(); ++b) c->drop_block(*b);
  c->by_admission.erase(it->second.admitted);
  c->seqs.erase(it);
  return PKV_OK;
}

int64_t pkv_cache_blocks_needed(pkv_cache* c, const int64_t* seq_ids, const int32_t* counts,
                                int32_t n) {
  if (!c || n < 0 || (n > 0 && (!seq_ids || !counts))) return -1;
  return c->plan(seq_ids, counts, n);
}

pkv_status pkv_cache_append(pkv_cache* c, const int64_t* seq_ids, const int32_t* counts,
                            int32_t n, int64_t* slot_mapping, int64_t slot_capacity,
                            int32_t* copies, int32_t copy_capacity, int64_t* num_slots,
                            int32_t* num_copies) {
  if (!c || n < 0 || !num_slots || !num_copies) return PKV_ERR_INVALID_ARG;
  *num_slots = 0;
  *num_copies = 0;
  if (n == 0) return PKV_OK;
  if (!seq_ids || !counts) return PKV_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int32_t i = 0; i < n; ++i) total += counts[i] > 0 ? counts[i] : 0;
  const int64_t need = c->plan(seq_ids, counts, n);
  if (need < 0) return PKV_ERR_INVALID_ARG;
  // each sequence copies at most one block per call (only its last, partly
  // filled page can be shared), so n pairs always suffice
  if (total > slot_capacity || (total > 0 && !slot_mapping)) return PKV_ERR_INVALID_ARG;
  if (copy_capacity < n || !copies) return PKV_ERR_INVALID_ARG;
  if (need > int64_t(c->free_stack.size())) return PKV_ERR_OUT_OF_BLOCKS;
  const int32_t P = c->block_size;
  int64_t k = 0;
  int32_t ncp = 0;
  for (int32_t i = 0; i < n; ++i) {
    pkv_cache::Seq& s = c->seqs.find(seq_ids[i])->second;
    for (int32_t t = 0; t < counts[i]; ++t) {
      const int32_t pos = s.len;
      const size_t j = size_t(pos / P);
      if (j == s.pages.size()) {
        s.pages.push_back(c->pop_block());
      } else if (c->owners[s.pages[j]] > 1) {
        const int32_t old = s.pages[j];
        const int32_t fresh = c->pop_block();
        --c->owners[old];
        s.pages[j] = fresh;
        copies[2 * ncp] = old;
        copies[2 * ncp + 1] = fresh;
        ++ncp;
      }
      slot_mapping[k++] = int64_t(s.pages[j]) * P + pos % P;
      s.len = pos + 1;
    }
  }
  *num_slots = k;
  *num_copies = ncp;
  return PKV_OK;
}

pkv_status pkv_cache_preempt_for(pkv_cache* c, int32_t needed, const int64_t* protected_ids,
                                 int32_t num_protected, int64_t* victims,
                                 int32_t victim_capacity, int32_t* num_victims) {
  if (!c || needed < 0 || num_protected < 0 || !num_victims ||
      (num_protected > 0 && !protected_ids))
    return PKV_ERR_INVALID_ARG;
  *num_victims = 0;
  std::unordered_set<int64_t> prot(protected_ids, protected_ids + num_protected);
  int64_t free_now = int64_t(c->free_stack.size());
  std::vector<int64_t> chosen;
  for (auto it = c->by_admission.rbegin(); it != c->by_admission.rend(); ++it) {
    if (free_now >= needed) break;
    if (prot.count(it->second)) continue;
    for (int32_t b : c->seqs.find(it->second)->second.pages) {
      c->add_delta(b, -1);
      if (c->owners[b] + c->delta[b] == 0) ++free_now;
    }
    chosen.push_back(it->second);
  }
  c->reset_delta();
  if (free_now < needed) return PKV_ERR_OUT_OF_BLOCKS;
  if (int64_t(chosen.size()) > victim_capacity || (!chosen.empty() && !victims))
    return PKV_ERR_INVALID_ARG;
  for (size_t i = 0; i < chosen.size(); ++i) {
    victims[i] = chosen[i];
    pkv_cache_release(c, chosen[i]);
  }
  *num_victims = int32_t(chosen.size());
  return PKV_OK;
}

pkv_status pkv_cache_block_tables(const pkv_cache* c, const int64_t* seq_ids, int32_t n,
                                  int32_t* block_tables, int32_t* context_lens) {
  if (!c || n < 0 || (n > 0 && (!seq_ids || !block_tables || !context_lens)))
    return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!c->seqs.count(seq_ids[i])) return PKV_ERR_INVALID_ARG;
  const int32_t M = c->max_blocks;
  for (int32_t i = 0; i < n; ++i) {
    const pkv_cache::Seq& s = c->seqs.find(seq_ids[i])->second;
    int32_t* row = block_tables + int64_t(i) * M;
    const int32_t np = int32_t(s.pages.size());
    for (int32_t j = 0; j < np; ++j) row[j] = s.pages[size_t(j)];
    for (int32_t j = np; j < M; ++j) row[j] = -1;
    context_lens[i] = s.len;
  }
  return PKV_OK;
}

}  // extern "C"
