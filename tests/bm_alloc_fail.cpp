// Allocation-failure injection for the host block manager (built and run by
// test_block_manager.py with the system C++ compiler; no GPU).
//
// The global operator new is replaced by one that can be told to fail at its
// k-th call.  Every call of a scripted sequence of operations is run with
// k = 0, 1, 2, ... until it completes without an injected failure; each
// injected failure must come back as PA_ERR_OOM (nullptr from create, -1 from
// the waste count) and leave every observable part of the manager -- free
// counts, reference counts, cached-block count, sequence lengths and block
// tables -- exactly as it was before the call.  Prints "ok <failures>".
#include <cstdio>
#include <cstdlib>
#include <functional>
#include <new>
#include <vector>

#include "pagedattn.h"

static long g_countdown = -1;  // allocations left before one fails; -1 = never
static bool g_fired = false;

void *operator new(std::size_t n) {
  if (g_countdown == 0) {
    g_countdown = -1;
    g_fired = true;
    throw std::bad_alloc();
  }
  if (g_countdown > 0) --g_countdown;
  void *p = std::malloc(n ? n : 1);
  if (!p) throw std::bad_alloc();
  return p;
}
void *operator new[](std::size_t n) { return operator new(n); }
void *operator new(std::size_t n, const std::nothrow_t &) noexcept {
  try {
    return operator new(n);
  } catch (...) {
    return nullptr;
  }
}
void operator delete(void *p) noexcept { std::free(p); }
void operator delete[](void *p) noexcept { std::free(p); }
void operator delete(void *p, std::size_t) noexcept { std::free(p); }
void operator delete[](void *p, std::size_t) noexcept { std::free(p); }

namespace {

constexpr int kBlocks = 48, kHost = 16, kB = 4, kSeqs = 8;

struct Snap {
  int nfree, ncached, nhost;
  std::vector<int> refs, lens;
  std::vector<std::vector<int32_t>> tables;
  bool operator==(const Snap &o) const {
    return nfree == o.nfree && ncached == o.ncached && nhost == o.nhost && refs == o.refs && lens == o.lens &&
           tables == o.tables;
  }
};

Snap snap(const pa_bm *bm) {
  Snap s;
  s.nfree = pa_bm_num_free(bm);
  s.ncached = pa_bm_num_cached_blocks(bm);
  s.nhost = pa_bm_num_free_host(bm);
  for (int b = 0; b < kBlocks; ++b) s.refs.push_back(pa_bm_ref_count(bm, b));
  for (int q = 0; q < kSeqs; ++q) {
    s.lens.push_back(pa_bm_seq_len(bm, q));
    std::vector<int32_t> t(256);
    int n = 0;
    if (pa_bm_block_table(bm, q, t.data(), (int)t.size(), &n) == PA_OK)
      t.resize(n);
    else
      t.clear();
    s.tables.push_back(t);
  }
  return s;
}

int failures = 0;

// Runs op with the k-th allocation failing, k = 0, 1, ..., until it completes.
// op returns its status; `oom` is the status that stands for a failed allocation.
bool inject(const char *name, pa_bm *bm, const std::function<long long()> &op, long long oom) {
  for (long k = 0;; ++k) {
    const Snap before = snap(bm);
    g_fired = false;
    g_countdown = k;
    const long long st = op();
    g_countdown = -1;
    if (!g_fired) return true;
    ++failures;
    if (st != oom) {
      std::printf("%s: allocation %ld failed, status %lld (want %lld)\n", name, k, st, oom);
      return false;
    }
    if (!(snap(bm) == before)) {
      std::printf("%s: allocation %ld failed and changed the state\n", name, k);
      return false;
    }
  }
}

}  // namespace

int main() {
  // creation: a failed allocation returns nullptr
  for (long k = 0;; ++k) {
    g_fired = false;
    g_countdown = k;
    pa_bm *bm = pa_bm_create_with_host(kBlocks, kHost, kB);
    g_countdown = -1;
    if (!g_fired) {
      pa_bm_destroy(bm);
      break;
    }
    ++failures;
    if (bm) {
      std::printf("create: allocation %ld failed but a manager came back\n", k);
      return 1;
    }
  }
  pa_bm *bm = pa_bm_create_with_host(kBlocks, kHost, kB);
  if (!bm) return 1;
  std::vector<int32_t> p(22), r(13);
  for (int i = 0; i < (int)p.size(); ++i) p[i] = 1000 + i;
  for (int i = 0; i < (int)r.size(); ++i) r[i] = 1000 + i;  // the first 3 blocks of p, then a tail
  r[12] = 7;
  int cached = 0;
  int64_t slot = 0, cow[2], pairs[2 * 64];
  int n = 0;
  const long long OOM = PA_ERR_OOM;
  bool ok = true;
  ok = ok && inject("add_seq_tokens (first prompt)", bm, [&] { return (long long)pa_bm_add_seq_tokens(bm, 0, p.data(), (int)p.size(), &cached); }, OOM);
  ok = ok && inject("add_seq_tokens (prefix hit)", bm, [&] { return (long long)pa_bm_add_seq_tokens(bm, 1, r.data(), (int)r.size(), &cached); }, OOM);
  ok = ok && inject("fork", bm, [&] { return (long long)pa_bm_fork(bm, 0, 2); }, OOM);
  for (int i = 0; i < 6 && ok; ++i)
    ok = inject("append (copy on write, new blocks)", bm, [&] { return (long long)pa_bm_append(bm, 2, &slot, cow); }, OOM);
  ok = ok && inject("add_seq", bm, [&] { return (long long)pa_bm_add_seq(bm, 3, 9); }, OOM);
  for (int i = 0; i < 40 && ok; ++i)
    ok = inject("append (growing table)", bm, [&] { return (long long)pa_bm_append(bm, 3, &slot, cow); }, OOM);
  for (int i = 0; i < 7 && ok; ++i) {  // seq 1 keeps its ids: fills and registers its block
    const int32_t tok = 500 + i;
    ok = inject("append_token", bm, [&] { return (long long)pa_bm_append_token(bm, 1, tok, &slot, cow); }, OOM);
  }
  ok = ok && pa_bm_fork(bm, 2, 5) == PA_OK;
  const int32_t ids[4] = {5, 0, 2, 3};
  int64_t bslots[4], bcows[8];
  for (int i = 0; i < 6 && ok; ++i)
    ok = inject("append_batch", bm, [&] { return (long long)pa_bm_append_batch(bm, ids, nullptr, 4, bslots, bcows); }, OOM);
  const int32_t tids[2] = {1, 0}, toks[2] = {900, 901};
  for (int i = 0; i < 5 && ok; ++i)
    ok = inject("append_batch (ids)", bm, [&] { return (long long)pa_bm_append_batch(bm, tids, toks, 2, bslots, bcows); }, OOM);
  ok = ok && inject("swap_out", bm, [&] { return (long long)pa_bm_swap_out(bm, 3, pairs, 64, &n); }, OOM);
  ok = ok && inject("wasted_slots", bm, [&] { return (long long)pa_bm_wasted_slots(bm); }, -1);
  ok = ok && inject("swap_in", bm, [&] { return (long long)pa_bm_swap_in(bm, 3, pairs, 64, &n); }, OOM);
  ok = ok && inject("free_seq", bm, [&] { return (long long)pa_bm_free_seq(bm, 0); }, OOM);
  ok = ok && inject("free_seq (fork)", bm, [&] { return (long long)pa_bm_free_seq(bm, 2); }, OOM);
  ok = ok && inject("add_seq_tokens (revived blocks)", bm, [&] { return (long long)pa_bm_add_seq_tokens(bm, 4, p.data(), (int)p.size(), &cached); }, OOM);
  if (ok && cached != 20) {
    std::printf("revived prompt found %d cached tokens, want 20\n", cached);
    ok = false;
  }
  for (int q : {1, 3, 4, 5})
    if (ok) ok = pa_bm_free_seq(bm, q) == PA_OK;
  if (ok && (pa_bm_num_free(bm) != kBlocks || pa_bm_num_free_host(bm) != kHost)) {
    std::printf("blocks lost: %d free of %d, %d host of %d\n", pa_bm_num_free(bm), kBlocks, pa_bm_num_free_host(bm),
                kHost);
    ok = false;
  }
  pa_bm_destroy(bm);
  if (!ok) return 1;
  std::printf("ok %d\n", failures);
  return 0;
}
