// Host block manager: O(1) free list, per-block refcounts, fork, append with
// copy-on-write, free.
//
// Rules ("PagedAttention: How vLLM Borrowed Virtual Memory to Unlock GPU Serving
// at Scale", sections "The OS-Inspired Insight" and "Walking Through the
// Lifecycle"; "What is paged attention?", section "How it works"):
//   * the pool is a fixed set of num_blocks blocks; alloc pops the free stack,
//     a block whose refcount drops to zero is pushed back;
//   * a sequence's block table maps logical block j to a physical id;
//   * position p needs a new block when p % B == 0; a write into a shared
//     (refcount > 1) partial last block first moves the writer onto a private
//     copy; slot(p) = table[p / B] * B + p % B;
//   * preemption by swapping ("PagedAttention — how vLLM stopped wasting 80% of
//     your GPU memory", section "Preemption: what happens when memory runs out
//     anyway"): swap-out hands back the sequence's blocks (their contents go to
//     host memory) and keeps its length; swap-in gives it ceil(len / B) fresh
//     blocks, all or nothing.
// Every public call validates first and mutates only once it cannot fail, so a
// failing call leaves the state unchanged.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <exception>
#include <memory>
#include <new>
#include <utility>
#include <vector>

#include "pkv.h"
#include "status.h"

namespace {

// Runs the body of an entry point that may allocate host memory; a failed
// allocation becomes an error code, so no C++ exception crosses the C ABI.  The
// bodies allocate before they change any state, so such a failure leaves the
// state unchanged like every other failing call.
template <typename F>
int guarded(F&& body) {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return pkv::fail(PKV_ERR_INVALID_ARG, "host memory exhausted");
  } catch (const std::exception& e) {
    return pkv::fail(PKV_ERR_INVALID_ARG, "host error: %s", e.what());
  }
}

// Makes room for `extra` more entries (growing geometrically), so that the
// push_backs which follow cannot allocate.
void ensure_room(std::vector<int32_t>& v, size_t extra) {
  if (v.size() + extra > v.capacity()) v.reserve(std::max(v.size() + extra, 2 * v.capacity()));
}

}  // namespace

struct pkv_allocator {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;   // back() is the next block handed out
  std::vector<int32_t> refcount;     // per physical block
  struct Seq {
    std::vector<int32_t> table;
    int32_t len = 0;
    bool live = false;
    bool swapped = false;  // blocks handed back by swap-out, not yet swapped in
    uint32_t mark = 0;     // batched append: the call that last listed it
  };
  std::vector<Seq> seqs;             // indexed by sequence id
  uint32_t mark_epoch = 0;           // batched append: calls so far

  bool valid_block(int32_t b) const { return b >= 0 && b < num_blocks; }
  bool allocated(int32_t b) const { return valid_block(b) && refcount[b] > 0; }
  bool live_seq(int32_t s) const {
    return s >= 0 && s < static_cast<int32_t>(seqs.size()) && seqs[s].live;
  }
  bool resident_seq(int32_t s) const { return live_seq(s) && !seqs[s].swapped; }

  int32_t pop() {
    int32_t b = free_stack.back();
    free_stack.pop_back();
    refcount[b] = 1;
    return b;
  }
  void decref(int32_t b) {
    if (--refcount[b] == 0) free_stack.push_back(b);
  }
  // Blocks an append of n tokens needs from the free list.
  int64_t needed(const Seq& s, int32_t n) const {
    if (n <= 0) return 0;
    const int64_t B = block_size;
    const int64_t t = s.len;
    const int64_t have = (t + B - 1) / B;
    const int64_t want = (t + n + B - 1) / B;
    int64_t need = want - have;
    if (t % B != 0 && refcount[s.table.back()] > 1) need += 1;  // copy-on-write of the partial block
    return need;
  }
};

extern "C" {

int pkv_allocator_create(int32_t num_blocks, int32_t block_size, const int32_t* pop_order,
                         pkv_allocator_t** out) {
  PKV_REQUIRE(out != nullptr, PKV_ERR_INVALID_ARG, "out is NULL");
  PKV_REQUIRE(num_blocks > 0 && block_size > 0, PKV_ERR_INVALID_ARG,
              "num_blocks (%d) and block_size (%d) must be positive", num_blocks, block_size);
  PKV_REQUIRE(static_cast<int64_t>(num_blocks) * block_size < (int64_t(1) << 31),
              PKV_ERR_INVALID_ARG, "num_blocks * block_size must be < 2^31");
  return guarded([&] {
    std::vector<int32_t> order(num_blocks);
    if (pop_order) {
      std::vector<char> seen(num_blocks, 0);
      for (int32_t i = 0; i < num_blocks; ++i) {
        int32_t b = pop_order[i];
        PKV_REQUIRE(b >= 0 && b < num_blocks && !seen[b], PKV_ERR_INVALID_ARG,
                    "pop_order is not a permutation of 0..%d (entry %d = %d)", num_blocks - 1, i,
                    b);
        seen[b] = 1;
        order[i] = b;
      }
    } else {
      for (int32_t i = 0; i < num_blocks; ++i) order[i] = i;
    }
    std::unique_ptr<pkv_allocator> a(new pkv_allocator());
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->free_stack.assign(order.rbegin(), order.rend());
    a->refcount.assign(num_blocks, 0);
    *out = a.release();
    return pkv::ok();
  });
}

int pkv_allocator_destroy(pkv_allocator_t* a) {
  delete a;
  return pkv::ok();
}

int pkv_block_alloc(pkv_allocator_t* a, int32_t* block_id) {
  PKV_REQUIRE(a && block_id, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(!a->free_stack.empty(), PKV_ERR_OUT_OF_BLOCKS, "no free block");
  *block_id = a->pop();
  return pkv::ok();
}

int pkv_block_incref(pkv_allocator_t* a, int32_t b) {
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL handle");
  PKV_REQUIRE(a->allocated(b), PKV_ERR_INVALID_ARG, "incref of unallocated block %d", b);
  a->refcount[b] += 1;
  return pkv::ok();
}

int pkv_block_decref(pkv_allocator_t* a, int32_t b) {
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL handle");
  PKV_REQUIRE(a->allocated(b), PKV_ERR_INVALID_ARG, "decref of unallocated block %d", b);
  a->decref(b);
  return pkv::ok();
}

int pkv_block_refcount(pkv_allocator_t* a, int32_t b, int32_t* rc) {
  PKV_REQUIRE(a && rc, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->valid_block(b), PKV_ERR_INVALID_ARG, "block %d out of range", b);
  *rc = a->refcount[b];
  return pkv::ok();
}

int pkv_num_free_blocks(pkv_allocator_t* a, int32_t* n) {
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  *n = static_cast<int32_t>(a->free_stack.size());
  return pkv::ok();
}

int pkv_seq_create(pkv_allocator_t* a, int32_t* seq) {
  PKV_REQUIRE(a && seq, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->seqs.size() < static_cast<size_t>(INT32_MAX), PKV_ERR_INVALID_ARG,
              "sequence ids exhausted");
  return guarded([&] {
    a->seqs.emplace_back();  // no effect if it throws
    a->seqs.back().live = true;
    *seq = static_cast<int32_t>(a->seqs.size() - 1);
    return pkv::ok();
  });
}

int pkv_seq_fork(pkv_allocator_t* a, int32_t parent, int32_t* child) {
  PKV_REQUIRE(a && child, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->resident_seq(parent), PKV_ERR_INVALID_ARG,
              "unknown or swapped-out sequence %d", parent);
  PKV_REQUIRE(a->seqs.size() < static_cast<size_t>(INT32_MAX), PKV_ERR_INVALID_ARG,
              "sequence ids exhausted");
  return guarded([&] {
    pkv_allocator::Seq c;
    c.table = a->seqs[parent].table;
    c.len = a->seqs[parent].len;
    c.live = true;
    a->seqs.push_back(std::move(c));  // no effect if it throws
    for (int32_t b : a->seqs.back().table) a->refcount[b] += 1;
    *child = static_cast<int32_t>(a->seqs.size() - 1);
    return pkv::ok();
  });
}

int pkv_seq_free(pkv_allocator_t* a, int32_t seq) {
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL handle");
  PKV_REQUIRE(a->live_seq(seq), PKV_ERR_INVALID_ARG, "unknown sequence %d", seq);
  auto& s = a->seqs[seq];
  for (auto it = s.table.rbegin(); it != s.table.rend(); ++it) a->decref(*it);
  s.table.clear();
  s.table.shrink_to_fit();
  s.len = 0;
  s.live = false;
  s.swapped = false;
  return pkv::ok();
}

int pkv_seq_swap_out(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity,
                     int32_t* n) {
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->resident_seq(seq), PKV_ERR_INVALID_ARG, "unknown or swapped-out sequence %d",
              seq);
  auto& s = a->seqs[seq];
  const int32_t m = static_cast<int32_t>(s.table.size());
  PKV_REQUIRE(m == 0 || (ids_out && capacity >= m), PKV_ERR_INVALID_ARG,
              "ids_out holds %d ids, the sequence has %d blocks", capacity, m);
  if (m) std::memcpy(ids_out, s.table.data(), sizeof(int32_t) * m);
  for (auto it = s.table.rbegin(); it != s.table.rend(); ++it) a->decref(*it);
  s.table.clear();
  s.swapped = true;
  *n = m;
  return pkv::ok();
}

int pkv_seq_swap_in(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity,
                    int32_t* n) {
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->live_seq(seq) && a->seqs[seq].swapped, PKV_ERR_INVALID_ARG,
              "sequence %d is not swapped out", seq);
  auto& s = a->seqs[seq];
  const int64_t B = a->block_size;
  const int32_t m = static_cast<int32_t>((s.len + B - 1) / B);
  PKV_REQUIRE(m == 0 || (ids_out && capacity >= m), PKV_ERR_INVALID_ARG,
              "ids_out holds %d ids, the sequence needs %d blocks", capacity, m);
  PKV_REQUIRE(static_cast<size_t>(m) <= a->free_stack.size(), PKV_ERR_OUT_OF_BLOCKS,
              "swap-in needs %d blocks, %zu free", m, a->free_stack.size());
  return guarded([&] {
    s.table.resize(m);  // before any block is taken; no effect if it throws
    for (int32_t j = 0; j < m; ++j) s.table[j] = ids_out[j] = a->pop();
    s.swapped = false;
    *n = m;
    return pkv::ok();
  });
}

int pkv_seq_blocks_needed(pkv_allocator_t* a, int32_t seq, int32_t n, int32_t* needed) {
  PKV_REQUIRE(a && needed, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->resident_seq(seq), PKV_ERR_INVALID_ARG, "unknown or swapped-out sequence %d",
              seq);
  PKV_REQUIRE(n >= 0, PKV_ERR_INVALID_ARG, "negative token count");
  *needed = static_cast<int32_t>(a->needed(a->seqs[seq], n));
  return pkv::ok();
}

int pkv_seq_append(pkv_allocator_t* a, int32_t seq, int32_t n, int32_t* slots_out,
                   int32_t* cow_pair_out, int32_t* n_cow) {
  PKV_REQUIRE(a && n_cow, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->resident_seq(seq), PKV_ERR_INVALID_ARG, "unknown or swapped-out sequence %d",
              seq);
  PKV_REQUIRE(n >= 0, PKV_ERR_INVALID_ARG, "negative token count");
  PKV_REQUIRE(n == 0 || slots_out, PKV_ERR_INVALID_ARG, "slots_out is NULL");
  auto& s = a->seqs[seq];
  const int64_t B = a->block_size;
  PKV_REQUIRE(static_cast<int64_t>(s.len) + n < (int64_t(1) << 31), PKV_ERR_INVALID_ARG,
              "sequence length overflow");
  const int64_t need = a->needed(s, n);
  PKV_REQUIRE(need <= static_cast<int64_t>(a->free_stack.size()), PKV_ERR_OUT_OF_BLOCKS,
              "append of %d tokens needs %lld blocks, %zu free", n, static_cast<long long>(need),
              a->free_stack.size());
  PKV_REQUIRE(need == 0 || cow_pair_out || !(s.len % B != 0 && a->refcount[s.table.back()] > 1),
              PKV_ERR_INVALID_ARG, "cow_pair_out is NULL but the append needs a copy");
  const int rc = guarded([&] {
    ensure_room(s.table, static_cast<size_t>(need));  // the loop below then cannot allocate
    return pkv::ok();
  });
  if (rc != PKV_OK) return rc;
  *n_cow = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t p = s.len;
    if (p % B == 0) {
      s.table.push_back(a->pop());
    } else if (a->refcount[s.table.back()] > 1) {
      const int32_t old_id = s.table.back();
      const int32_t new_id = a->pop();
      cow_pair_out[0] = old_id;
      cow_pair_out[1] = new_id;
      *n_cow = 1;
      a->decref(old_id);
      s.table.back() = new_id;
    }
    slots_out[i] = static_cast<int32_t>(s.table[p / B] * B + p % B);
    s.len = static_cast<int32_t>(p + 1);
  }
  return pkv::ok();
}

int pkv_seq_append_one_each(pkv_allocator_t* a, const int32_t* seqs, int32_t k,
                            int32_t* slots_out, int32_t* cow_pairs_out, int32_t* n_cow) {
  PKV_REQUIRE(a && n_cow, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(k >= 0, PKV_ERR_INVALID_ARG, "negative sequence count");
  PKV_REQUIRE(k == 0 || (seqs && slots_out && cow_pairs_out), PKV_ERR_INVALID_ARG,
              "NULL array");
  return guarded([&] {
    const int64_t B = a->block_size;
    // validate every sequence, and count the blocks the appends take in order: a
    // copy-on-write earlier in the list may leave a later sequence the last holder
    // of its block, which it then writes in place
    std::vector<std::pair<int32_t, int32_t>> drops;  // (block, refcount dropped so far)
    int64_t need = 0;
    // a sequence listed twice is found by its mark (this call's number), in O(k)
    if (++a->mark_epoch == 0) {
      for (auto& s : a->seqs) s.mark = 0;
      a->mark_epoch = 1;
    }
    const uint32_t epoch = a->mark_epoch;
    for (int32_t i = 0; i < k; ++i) {
      const int32_t q = seqs[i];
      PKV_REQUIRE(a->resident_seq(q), PKV_ERR_INVALID_ARG, "unknown or swapped-out sequence %d",
                  q);
      PKV_REQUIRE(a->seqs[q].mark != epoch, PKV_ERR_INVALID_ARG, "sequence %d listed twice", q);
      a->seqs[q].mark = epoch;
      auto& s = a->seqs[q];
      PKV_REQUIRE(s.len < INT32_MAX, PKV_ERR_INVALID_ARG, "sequence length overflow");
      if (s.len % B == 0) {
        ++need;
        ensure_room(s.table, 1);  // its push_back below then cannot allocate
        continue;
      }
      const int32_t last = s.table.back();
      int32_t rc = a->refcount[last];
      size_t d = 0;
      while (d < drops.size() && drops[d].first != last) ++d;
      if (d < drops.size()) rc -= drops[d].second;
      if (rc > 1) {
        ++need;
        if (d < drops.size()) ++drops[d].second; else drops.emplace_back(last, 1);
      }
    }
    PKV_REQUIRE(need <= static_cast<int64_t>(a->free_stack.size()), PKV_ERR_OUT_OF_BLOCKS,
                "appending one token to each of %d sequences needs %lld blocks, %zu free", k,
                static_cast<long long>(need), a->free_stack.size());
    int32_t nc = 0;
    for (int32_t i = 0; i < k; ++i) {
      auto& s = a->seqs[seqs[i]];
      const int64_t p = s.len;
      if (p % B == 0) {
        s.table.push_back(a->pop());
      } else if (a->refcount[s.table.back()] > 1) {
        const int32_t old_id = s.table.back();
        const int32_t new_id = a->pop();
        cow_pairs_out[2 * nc] = old_id;
        cow_pairs_out[2 * nc + 1] = new_id;
        ++nc;
        a->decref(old_id);
        s.table.back() = new_id;
      }
      slots_out[i] = static_cast<int32_t>(s.table[p / B] * B + p % B);
      s.len = static_cast<int32_t>(p + 1);
    }
    *n_cow = nc;
    return pkv::ok();
  });
}

int pkv_seq_len(pkv_allocator_t* a, int32_t seq, int32_t* len) {
  PKV_REQUIRE(a && len, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->live_seq(seq), PKV_ERR_INVALID_ARG, "unknown sequence %d", seq);
  *len = a->seqs[seq].len;
  return pkv::ok();
}

int pkv_seq_table(pkv_allocator_t* a, int32_t seq, int32_t* ids_out, int32_t capacity,
                  int32_t* n) {
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->live_seq(seq), PKV_ERR_INVALID_ARG, "unknown sequence %d", seq);
  PKV_REQUIRE(capacity >= 0 && (capacity == 0 || ids_out), PKV_ERR_INVALID_ARG,
              "bad output buffer");
  const auto& t = a->seqs[seq].table;
  const int32_t m = static_cast<int32_t>(t.size());
  const int32_t c = m < capacity ? m : capacity;
  if (c > 0) std::memcpy(ids_out, t.data(), sizeof(int32_t) * c);
  *n = m;
  return pkv::ok();
}

int pkv_export_tables(pkv_allocator_t* a, const int32_t* seqs, int32_t num, int32_t max_blocks,
                      int32_t* tables_out, int32_t* ctx_out) {
  PKV_REQUIRE(a && (num == 0 || (seqs && tables_out && ctx_out)), PKV_ERR_INVALID_ARG,
              "NULL argument");
  PKV_REQUIRE(num >= 0 && max_blocks >= 0, PKV_ERR_INVALID_ARG, "negative size");
  for (int32_t r = 0; r < num; ++r) {
    PKV_REQUIRE(a->resident_seq(seqs[r]), PKV_ERR_INVALID_ARG,
                "unknown or swapped-out sequence %d", seqs[r]);
    PKV_REQUIRE(a->seqs[seqs[r]].table.size() <= static_cast<size_t>(max_blocks),
                PKV_ERR_INVALID_ARG, "table of sequence %d has %zu blocks > max_blocks %d",
                seqs[r], a->seqs[seqs[r]].table.size(), max_blocks);
  }
  for (int32_t r = 0; r < num; ++r) {
    const auto& s = a->seqs[seqs[r]];
    int32_t* row = tables_out + static_cast<int64_t>(r) * max_blocks;
    const size_t m = s.table.size();
    if (m) std::memcpy(row, s.table.data(), sizeof(int32_t) * m);
    for (int32_t j = static_cast<int32_t>(m); j < max_blocks; ++j) row[j] = 0;
    ctx_out[r] = s.len;
  }
  return pkv::ok();
}

}  // extern "C"
