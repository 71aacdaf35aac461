// Paged KV-cache page allocator with refcounted prefix sharing (host side).
//
// Pages hold `page_size` consecutive token positions of every layer's keys
// and values. A sequence's block table lists its pages in position order:
// entry i covers positions [i*P, (i+1)*P). Pages shared from a registered
// prompt prefix ("OCRia-1 technical report guide", inference stack: reuse of
// the shared prompt prefix) come first and are refcounted, so a sequence
// releases them without freeing pages other sequences still read.
//
// The allocator is plain host C++ with no CUDA dependency; the model keeps
// the device copy of the block tables in step with it.
#pragma once
#include <cstdint>
#include <vector>

namespace spec {

enum { POOL_OK = 0, POOL_ERR_ARG = -1, POOL_ERR_NO_PAGES = -2, POOL_ERR_STATE = -4 };

class KvPool {
 public:
  KvPool(int n_pages, int page_size, int n_slots, int max_pages_per_seq)
      : n_pages_(n_pages), P_(page_size), max_pps_(max_pages_per_seq),
        ref_(n_pages, 0), bt_(n_slots), len_(n_slots, 0) {
    free_.reserve(n_pages);
    for (int i = n_pages - 1; i >= 0; --i) free_.push_back(i);  // pop gives 0 first
  }

  int page_size() const { return P_; }
  int n_slots() const { return (int)bt_.size(); }
  int max_pages_per_seq() const { return max_pps_; }
  int free_count() const { return (int)free_.size(); }
  bool valid_seq(int s) const { return s >= 0 && s < (int)bt_.size(); }
  const std::vector<int32_t>& table(int s) const { return bt_[s]; }
  int length(int s) const { return len_[s]; }
  int refcount(int page) const { return (page >= 0 && page < n_pages_) ? ref_[page] : -1; }
  static int pages_for(int n_tokens, int P) { return (n_tokens + P - 1) / P; }

  // Ensure seq holds pages for positions [0, n_tokens). All-or-nothing.
  int reserve(int s, int n_tokens) {
    if (!valid_seq(s) || n_tokens < 0) return POOL_ERR_ARG;
    int need = pages_for(n_tokens, P_);
    if (need > max_pps_) return POOL_ERR_ARG;
    int add = need - (int)bt_[s].size();
    if (add <= 0) return POOL_OK;
    if (add > (int)free_.size()) return POOL_ERR_NO_PAGES;
    for (int i = 0; i < add; ++i) {
      int pg = free_.back();
      free_.pop_back();
      ref_[pg] = 1;
      bt_[s].push_back(pg);
    }
    return POOL_OK;
  }

  // Commit a new length: keep pages covering max(new_len, keep_pages * P)
  // positions and release the pages past that.
  int commit(int s, int new_len, int keep_pages) {
    if (!valid_seq(s) || new_len < 0) return POOL_ERR_ARG;
    int keep = pages_for(new_len, P_);
    if (keep_pages > keep) keep = keep_pages;
    if (pages_for(new_len, P_) > (int)bt_[s].size()) return POOL_ERR_STATE;
    while ((int)bt_[s].size() > keep) {
      unref(bt_[s].back());
      bt_[s].pop_back();
    }
    len_[s] = new_len;
    return POOL_OK;
  }

  void set_length(int s, int n) { len_[s] = n; }

  int release(int s) {
    if (!valid_seq(s)) return POOL_ERR_ARG;
    for (int pg : bt_[s]) unref(pg);
    bt_[s].clear();
    len_[s] = 0;
    return POOL_OK;
  }

  // dst (empty) takes references to the first n pages of src.
  int share(int src, int n, int dst) {
    if (!valid_seq(src) || !valid_seq(dst) || src == dst || n < 0) return POOL_ERR_ARG;
    if (n > (int)bt_[src].size() || !bt_[dst].empty()) return POOL_ERR_STATE;
    for (int i = 0; i < n; ++i) {
      int pg = bt_[src][i];
      ref_[pg] += 1;
      bt_[dst].push_back(pg);
    }
    return POOL_OK;
  }

  // Replace seq's table by `pages` (used to mirror a device-side trim).
  void truncate_table(int s, int n) {
    while ((int)bt_[s].size() > n) {
      unref(bt_[s].back());
      bt_[s].pop_back();
    }
  }

 private:
  void unref(int pg) {
    if (--ref_[pg] == 0) free_.push_back(pg);
  }
  int n_pages_, P_, max_pps_;
  std::vector<int32_t> ref_;
  std::vector<int32_t> free_;
  std::vector<std::vector<int32_t>> bt_;
  std::vector<int32_t> len_;
};

}  // namespace spec
