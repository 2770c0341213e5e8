// Work-conserving dispatch of GPU-bound API calls (the Pie review, section 5:
// Algorithm 2, Eq. (4), horizontal and vertical batching).  The policy, call by
// call, is stated in include/pie_batcher.h; this file holds the bookkeeping.
//
// Per call: queue, handler type, rows, working-set key, state (queued, in
// flight, done), dependencies and read/write sets as given (the Eq. (4) test
// marks and checks one stamp per resource, so neither order nor repeats matter).  Per
// queue: its priority and its queued calls in arrival order.  A dispatch walks
// the queues that hold calls (a list kept in insertion order, compacted as
// queues empty), builds each ready queue's group, buckets the groups by
// handler type, and for each type takes groups in priority order under Eq. (4)
// against the union of the read and write sets already taken (which is the
// same test as Eq. (4) against every taken group in turn), then truncates.
// Resource ids are small non-negative integers (KV page ids), so the taken
// sets are two arrays indexed by resource id holding the stamp of the last
// candidate that marked the resource: marking and testing cost one access.
//
// Forward calls on registered working sets: the batcher holds each working
// set's pages in slot order, derives a forward call's read set (the pages of
// every slot up to its last row's) and write set (the pages of its new
// slots) from them, and turns a dispatched batch into the pass's geometry
// (the folding geometry of "The forward pass", State geometry), so that no
// per-page list crosses the API boundary on the control loop's path.

#include <algorithm>
#include <cstring>
#include <deque>
#include <string>
#include <vector>

#include "internal.h"
#include "pie_batcher.h"

namespace {

using pie::set_last_error;

enum State : uint8_t { kQueued = 0, kInFlight = 1, kDone = 2 };

struct CallRec {
  int32_t queue, handler;
  int64_t rows, key;
  std::vector<int64_t> deps, reads, writes;
};

struct Queue {
  int32_t priority;
  std::deque<int64_t> ids;  // queued calls, arrival order
  bool listed = false;      // present in Batcher::active
};

struct Group {
  int32_t queue;
  std::vector<int64_t> ids;
};

constexpr int64_t kMaxResource = int64_t(1) << 26;  // resource ids: [0, 2^26)

}  // namespace

struct pie_batcher {
  std::vector<uint8_t> ordered;
  int32_t max_calls;
  int64_t max_rows;
  std::vector<CallRec> calls;
  std::vector<uint8_t> state;
  std::vector<Queue> queues;
  std::vector<int32_t> active;  // queues that may hold calls
  int64_t queued = 0, in_flight = 0;
  std::vector<uint32_t> rstamp, wstamp;  // per resource: stamp of the candidate that read / wrote it
  uint32_t stamp = 0;
  std::vector<std::vector<int32_t>> ws_pages;  // per working-set key: its pages in slot order
  std::vector<uint8_t> ws_known;               // per key: pages registered
  std::vector<int64_t> scratch;                // per-call read/write lists being built
  // the last planned pass's geometry (pie_batcher_plan_forward), kept until
  // the next one: row_indptr, positions, kv_len, page_indptr, page_ids, fold_mode
  std::vector<int32_t> pass_i32[6];

  // a new candidate: a fresh stamp (arrays cleared when the counter wraps)
  uint32_t next_stamp() {
    if (++stamp == 0) {
      std::fill(rstamp.begin(), rstamp.end(), 0u);
      std::fill(wstamp.begin(), wstamp.end(), 0u);
      stamp = 1;
    }
    return stamp;
  }

  bool ready(int64_t id) const {
    for (int64_t d : calls[size_t(id)].deps)
      if (state[size_t(d)] != kDone) return false;
    return true;
  }

  // the queue's ready head and its vertical group (Algorithm 2)
  void group_of(int32_t q, Group* g) const {
    g->queue = q;
    g->ids.clear();
    const Queue& Q = queues[size_t(q)];
    if (Q.ids.empty() || !ready(Q.ids.front())) return;
    const int64_t head = Q.ids.front();
    g->ids.push_back(head);
    const int32_t h = calls[size_t(head)].handler;
    if (!ordered[size_t(h)]) return;
    for (size_t i = 1; i < Q.ids.size(); ++i) {
      const CallRec& c = calls[size_t(Q.ids[i])];
      if (c.handler != h) break;
      bool ok = true;
      for (int64_t d : c.deps)
        if (state[size_t(d)] != kDone &&
            std::find(g->ids.begin(), g->ids.end(), d) == g->ids.end()) {
          ok = false;
          break;
        }
      if (!ok) break;
      g->ids.push_back(Q.ids[i]);
    }
  }
};

extern "C" {

int pie_batcher_create(int32_t num_handlers, const uint8_t* ordered, int32_t max_calls,
                       int64_t max_rows, pie_batcher_t** out) {
  if (!out) return set_last_error(PIE_EINVAL, "out is NULL");
  *out = nullptr;
  if (num_handlers < 1) return set_last_error(PIE_EINVAL, "num_handlers < 1");
  if (max_calls < 1 || max_rows < 1) return set_last_error(PIE_EINVAL, "batch limits must be >= 1");
  pie_batcher_t* b = new pie_batcher_t;
  b->ordered.assign(size_t(num_handlers), 0);
  if (ordered)
    for (int h = 0; h < num_handlers; ++h) b->ordered[size_t(h)] = ordered[h] ? 1 : 0;
  b->max_calls = max_calls;
  b->max_rows = max_rows;
  *out = b;
  return PIE_OK;
}

void pie_batcher_destroy(pie_batcher_t* b) { delete b; }

int pie_batcher_add_queue(pie_batcher_t* b, int32_t priority, int32_t* queue_id) {
  if (!b || !queue_id) return set_last_error(PIE_EINVAL, "NULL argument");
  if (b->queues.size() >= size_t(INT32_MAX)) return set_last_error(PIE_ERANGE, "too many queues");
  Queue q;
  q.priority = priority;
  b->queues.push_back(std::move(q));
  *queue_id = int32_t(b->queues.size() - 1);
  return PIE_OK;
}

}  // extern "C"

namespace {

// Checks one call that would get id `id`; on success *top is its largest
// resource id (-1 without any).
int check_call(const pie_batcher_t* b, int64_t id, int32_t queue, int32_t handler, int64_t rows,
               const int64_t* deps, int64_t num_deps, const int64_t* reads, int64_t num_reads,
               const int64_t* writes, int64_t num_writes, int64_t* top) {
  if (queue < 0 || size_t(queue) >= b->queues.size()) return set_last_error(PIE_EINVAL, "unknown queue");
  if (handler < 0 || size_t(handler) >= b->ordered.size())
    return set_last_error(PIE_EINVAL, "unknown handler type");
  if (rows < 1) return set_last_error(PIE_EINVAL, "rows < 1");
  if (num_deps < 0 || num_reads < 0 || num_writes < 0) return set_last_error(PIE_EINVAL, "negative count");
  if ((num_deps && !deps) || (num_reads && !reads) || (num_writes && !writes))
    return set_last_error(PIE_EINVAL, "NULL array with a positive count");
  for (int64_t i = 0; i < num_deps; ++i)
    if (deps[i] < 0 || deps[i] >= id)
      return set_last_error(PIE_EINVAL, "a dependency is not an earlier call");
  int64_t t = -1;
  for (int64_t i = 0; i < num_reads; ++i) t = reads[i] < 0 ? kMaxResource : std::max(t, reads[i]);
  for (int64_t i = 0; i < num_writes; ++i) t = writes[i] < 0 ? kMaxResource : std::max(t, writes[i]);
  if (t >= kMaxResource) return set_last_error(PIE_ERANGE, "resource id outside [0, 2^26)");
  *top = t;
  return PIE_OK;
}

// Records a checked call under the next id.
void add_call(pie_batcher_t* b, int64_t top, int32_t queue, int32_t handler, int64_t rows,
              int64_t key, const int64_t* deps, int64_t num_deps, const int64_t* reads,
              int64_t num_reads, const int64_t* writes, int64_t num_writes) {
  if (top >= int64_t(b->rstamp.size())) {
    const size_t n = std::max<size_t>(size_t(top) + 1, 2 * b->rstamp.size());
    b->rstamp.resize(n, 0u);
    b->wstamp.resize(n, 0u);
  }
  const int64_t id = int64_t(b->calls.size());
  CallRec c;
  c.queue = queue;
  c.handler = handler;
  c.rows = rows;
  c.key = key < 0 ? -1 : key;
  c.deps.assign(deps, deps + num_deps);
  c.reads.assign(reads, reads + num_reads);
  c.writes.assign(writes, writes + num_writes);
  b->calls.push_back(std::move(c));
  b->state.push_back(kQueued);
  Queue& Q = b->queues[size_t(queue)];
  Q.ids.push_back(id);
  if (!Q.listed) {
    Q.listed = true;
    b->active.push_back(queue);
  }
  ++b->queued;
}

// One flat list's entries of call i: [indptr[i], indptr[i+1]).
bool check_indptr(const int64_t* indptr, int32_t n, const int64_t* flat) {
  if (!indptr) return false;
  if (indptr[0] != 0) return false;
  for (int32_t i = 0; i < n; ++i)
    if (indptr[i + 1] < indptr[i]) return false;
  return indptr[n] == 0 || flat != nullptr;
}

}  // namespace

extern "C" {

int pie_batcher_submit(pie_batcher_t* b, int32_t queue, int32_t handler, int64_t rows,
                       int64_t key, const int64_t* deps, int32_t num_deps,
                       const int64_t* reads, int32_t num_reads, const int64_t* writes,
                       int32_t num_writes, int64_t* call_id) {
  if (!b || !call_id) return set_last_error(PIE_EINVAL, "NULL argument");
  int64_t top = -1;
  const int rc = check_call(b, int64_t(b->calls.size()), queue, handler, rows, deps, num_deps, reads,
                            num_reads, writes, num_writes, &top);
  if (rc != PIE_OK) return rc;
  *call_id = int64_t(b->calls.size());
  add_call(b, top, queue, handler, rows, key, deps, num_deps, reads, num_reads, writes, num_writes);
  return PIE_OK;
}

int pie_batcher_submit_many(pie_batcher_t* b, int32_t n, const int32_t* queues,
                            const int32_t* handlers, const int64_t* rows, const int64_t* keys,
                            const int64_t* dep_indptr, const int64_t* deps,
                            const int64_t* read_indptr, const int64_t* reads,
                            const int64_t* write_indptr, const int64_t* writes,
                            int64_t* first_id) {
  if (!b || !first_id || n < 0) return set_last_error(PIE_EINVAL, "NULL argument or n < 0");
  const int64_t id0 = int64_t(b->calls.size());
  *first_id = id0;
  if (n == 0) return PIE_OK;
  if (!queues || !handlers || !rows || !keys) return set_last_error(PIE_EINVAL, "NULL per-call array");
  if (!check_indptr(dep_indptr, n, deps) || !check_indptr(read_indptr, n, reads) ||
      !check_indptr(write_indptr, n, writes))
    return set_last_error(PIE_EINVAL, "a list offset array is NULL, not from 0 or decreasing");
  std::vector<int64_t> tops(size_t(n), -1);
  for (int32_t i = 0; i < n; ++i) {  // every call checked before any is recorded
    const int rc = check_call(b, id0 + i, queues[i], handlers[i], rows[i], deps + dep_indptr[i],
                              dep_indptr[i + 1] - dep_indptr[i], reads + read_indptr[i],
                              read_indptr[i + 1] - read_indptr[i], writes + write_indptr[i],
                              write_indptr[i + 1] - write_indptr[i], &tops[size_t(i)]);
    if (rc != PIE_OK) return rc;
  }
  for (int32_t i = 0; i < n; ++i)
    add_call(b, tops[size_t(i)], queues[i], handlers[i], rows[i], keys[i], deps + dep_indptr[i],
             dep_indptr[i + 1] - dep_indptr[i], reads + read_indptr[i],
             read_indptr[i + 1] - read_indptr[i], writes + write_indptr[i],
             write_indptr[i + 1] - write_indptr[i]);
  return PIE_OK;
}

int pie_batcher_dispatch(pie_batcher_t* b, int64_t* calls, int32_t* lanes, int32_t capacity,
                         int32_t* num_calls, int32_t* handler) {
  if (!b || !calls || !lanes || !num_calls || !handler)
    return set_last_error(PIE_EINVAL, "NULL argument");
  if (capacity < b->max_calls) return set_last_error(PIE_ENOSPACE, "capacity < max_calls");
  *num_calls = 0;
  *handler = -1;

  // ready groups, bucketed by handler type; drop empty queues
  std::vector<std::vector<Group>> by_type(b->ordered.size());
  size_t keep = 0;
  for (size_t i = 0; i < b->active.size(); ++i) {
    const int32_t q = b->active[i];
    Queue& Q = b->queues[size_t(q)];
    if (Q.ids.empty()) {
      Q.listed = false;
      continue;
    }
    b->active[keep++] = q;
    Group g;
    b->group_of(q, &g);
    if (!g.ids.empty()) by_type[size_t(b->calls[size_t(g.ids[0])].handler)].push_back(std::move(g));
  }
  b->active.resize(keep);

  // per handler type: priority order, Eq. (4) and the limits; then the oldest
  // call decides between handler types
  std::vector<std::pair<int32_t, std::vector<int64_t>>> best_batch;  // (group index, kept ids)
  int64_t best_oldest = -1;
  int32_t best_type = -1;
  std::vector<const Group*> order;
  for (size_t h = 0; h < by_type.size(); ++h) {
    std::vector<Group>& groups = by_type[h];
    if (groups.empty()) continue;
    order.clear();
    for (const Group& g : groups) order.push_back(&g);
    std::sort(order.begin(), order.end(), [&](const Group* u, const Group* v) {
      const int32_t pu = b->queues[size_t(u->queue)].priority;
      const int32_t pv = b->queues[size_t(v->queue)].priority;
      return pu != pv ? pu > pv : u->ids[0] < v->ids[0];
    });
    const uint32_t st = b->next_stamp();
    uint32_t* rs = b->rstamp.data();
    uint32_t* ws = b->wstamp.data();
    std::vector<std::pair<int32_t, std::vector<int64_t>>> cand;
    int64_t n_calls = 0, n_rows = 0, oldest = INT64_MAX;
    bool stop = false;
    for (size_t gi = 0; gi < order.size() && !stop; ++gi) {
      const Group& g = *order[gi];
      // Eq. (4) against every group taken so far: the group's writes meet no
      // taken read or write, its reads no taken write
      bool clash = false;
      for (size_t i = 0; i < g.ids.size() && !clash; ++i) {
        const CallRec& c = b->calls[size_t(g.ids[i])];
        for (int64_t x : c.writes)
          if (rs[x] == st || ws[x] == st) clash = true;
        for (int64_t x : c.reads)
          if (ws[x] == st) clash = true;
      }
      if (clash) continue;
      for (int64_t id : g.ids) {
        const CallRec& c = b->calls[size_t(id)];
        for (int64_t x : c.reads) rs[x] = st;
        for (int64_t x : c.writes) ws[x] = st;
      }
      std::vector<int64_t> kept;
      for (int64_t id : g.ids) {
        const int64_t rows = b->calls[size_t(id)].rows;
        if (n_calls > 0 && (n_calls + 1 > b->max_calls || n_rows + rows > b->max_rows)) {
          stop = true;
          break;
        }
        kept.push_back(id);
        ++n_calls;
        n_rows += rows;
        oldest = std::min(oldest, id);
      }
      if (!kept.empty()) cand.emplace_back(int32_t(gi), std::move(kept));
    }
    if (!cand.empty() && (best_type < 0 || oldest < best_oldest)) {
      best_oldest = oldest;
      best_type = int32_t(h);
      best_batch = std::move(cand);
    }
  }
  if (best_type < 0) return PIE_OK;

  // lanes, and the calls leave their queues (each group is its queue's prefix)
  int32_t n = 0, lane = -1;
  for (auto& kv : best_batch) {
    const std::vector<int64_t>& kept = kv.second;
    int64_t prev_key = -1;
    for (size_t i = 0; i < kept.size(); ++i) {
      const CallRec& c = b->calls[size_t(kept[i])];
      if (i == 0 || c.key < 0 || c.key != prev_key) ++lane;
      prev_key = c.key;
      calls[n] = kept[i];
      lanes[n] = lane;
      ++n;
    }
    Queue& Q = b->queues[size_t(b->calls[size_t(kept[0])].queue)];
    for (size_t i = 0; i < kept.size(); ++i) {
      Q.ids.pop_front();
      b->state[size_t(kept[i])] = kInFlight;
    }
  }
  b->queued -= n;
  b->in_flight += n;
  *num_calls = n;
  *handler = best_type;
  return PIE_OK;
}

int pie_batcher_complete(pie_batcher_t* b, const int64_t* calls, int32_t n) {
  if (!b || (n > 0 && !calls) || n < 0) return set_last_error(PIE_EINVAL, "bad arguments");
  for (int i = 0; i < n; ++i)
    if (calls[i] < 0 || size_t(calls[i]) >= b->state.size() || b->state[size_t(calls[i])] != kInFlight)
      return set_last_error(PIE_EINVAL, "a completed call was not in flight");
  for (int i = 0; i < n; ++i) {
    if (b->state[size_t(calls[i])] == kInFlight) {  // duplicates in the list count once
      b->state[size_t(calls[i])] = kDone;
      --b->in_flight;
      CallRec& c = b->calls[size_t(calls[i])];
      std::vector<int64_t>().swap(c.deps);  // no longer needed: only its state is read
      std::vector<int64_t>().swap(c.reads);
      std::vector<int64_t>().swap(c.writes);
    }
  }
  return PIE_OK;
}

int pie_batcher_set_pages(pie_batcher_t* b, int64_t key, const int32_t* pages, int32_t num_pages) {
  if (!b || num_pages < 0 || (num_pages > 0 && !pages))
    return set_last_error(PIE_EINVAL, "NULL batcher, negative count or NULL pages");
  if (key < 0 || key >= kMaxResource) return set_last_error(PIE_ERANGE, "key outside [0, 2^26)");
  for (int32_t i = 0; i < num_pages; ++i)
    if (pages[i] < 0 || pages[i] >= kMaxResource)
      return set_last_error(PIE_ERANGE, "page id outside [0, 2^26)");
  if (size_t(key) >= b->ws_pages.size()) {
    b->ws_pages.resize(size_t(key) + 1);
    b->ws_known.resize(size_t(key) + 1, 0);
  }
  b->ws_pages[size_t(key)].assign(pages, pages + num_pages);
  b->ws_known[size_t(key)] = 1;
  return PIE_OK;
}

int pie_batcher_submit_forward(pie_batcher_t* b, int32_t n, const int32_t* queues, int32_t handler,
                               const int64_t* keys, const int64_t* rows, const int64_t* first_slot,
                               int32_t page_size, int64_t* first_id) {
  if (!b || !first_id || n < 0) return set_last_error(PIE_EINVAL, "NULL argument or n < 0");
  const int64_t id0 = int64_t(b->calls.size());
  *first_id = id0;
  if (n == 0) return PIE_OK;
  if (!queues || !keys || !rows || !first_slot) return set_last_error(PIE_EINVAL, "NULL per-call array");
  if (page_size < 1) return set_last_error(PIE_EINVAL, "page_size < 1");
  // every call checked before any is recorded
  for (int32_t i = 0; i < n; ++i) {
    int64_t top = -1;
    const int rc = check_call(b, id0 + i, queues[i], handler, rows[i], nullptr, 0, nullptr, 0,
                              nullptr, 0, &top);
    if (rc != PIE_OK) return rc;
    const int64_t k = keys[i];
    if (k < 0 || size_t(k) >= b->ws_known.size() || !b->ws_known[size_t(k)])
      return set_last_error(PIE_EINVAL, "a call names a working set with no registered pages");
    const int64_t end = first_slot[i] + rows[i];  // one past the call's last slot
    if (first_slot[i] < 0 || end > int64_t(b->ws_pages[size_t(k)].size()) * page_size)
      return set_last_error(PIE_ERANGE, "a call's slots lie outside its working set's pages");
  }
  for (int32_t i = 0; i < n; ++i) {
    const std::vector<int32_t>& pg = b->ws_pages[size_t(keys[i])];
    const int64_t last = (first_slot[i] + rows[i] - 1) / page_size;  // page of the last new slot
    const int64_t w0 = first_slot[i] / page_size;
    // reads: the pages of slots [0, last slot]; writes: those of the new slots
    std::vector<int64_t>& r = b->scratch;
    r.assign(pg.begin(), pg.begin() + (last + 1));
    int64_t top = -1;
    for (int64_t x : r) top = std::max(top, x);
    add_call(b, top, queues[i], handler, rows[i], keys[i], nullptr, 0, r.data(), int64_t(r.size()),
             r.data() + w0, last + 1 - w0);
  }
  return PIE_OK;
}

int pie_batcher_forward_pass(const pie_batcher_t* b, const int64_t* calls, const int32_t* lanes,
                             int32_t n, const int32_t* frozen, int64_t num_keys, int32_t max_lanes,
                             int64_t max_rows, int64_t max_pages, int32_t* row_indptr,
                             int32_t* positions, int32_t* kv_len, int32_t* page_indptr,
                             int32_t* page_ids, int64_t* lane_keys, int32_t* first_row,
                             int32_t* num_lanes, int32_t* num_rows, int64_t* num_pages) {
  if (!b || n < 0 || (n > 0 && (!calls || !lanes || !frozen || !first_row)) || !num_lanes ||
      !num_rows || !num_pages)
    return set_last_error(PIE_EINVAL, "NULL argument or n < 0");
  int32_t L = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (calls[i] < 0 || size_t(calls[i]) >= b->calls.size())
      return set_last_error(PIE_EINVAL, "unknown call id");
    if (lanes[i] < 0 || lanes[i] >= n) return set_last_error(PIE_EINVAL, "lane outside [0, n)");
    L = std::max(L, lanes[i] + 1);
  }
  // each lane's working set and rows; a working set in one lane only
  std::vector<int64_t> key(size_t(L), -1), lrows(size_t(L), 0);
  for (int32_t i = 0; i < n; ++i) {
    const CallRec& c = b->calls[size_t(calls[i])];
    const int32_t l = lanes[i];
    if (c.key < 0 || size_t(c.key) >= b->ws_known.size() || !b->ws_known[size_t(c.key)] ||
        c.key >= num_keys)
      return set_last_error(PIE_EINVAL, "a call's working set has no registered pages or frozen length");
    if (key[size_t(l)] >= 0 && key[size_t(l)] != c.key)
      return set_last_error(PIE_EINVAL, "a lane of the batch spans two working sets");
    key[size_t(l)] = c.key;
    lrows[size_t(l)] += c.rows;
  }
  int64_t N = 0, NP = 0;
  for (int32_t l = 0; l < L; ++l) {
    if (key[size_t(l)] < 0) return set_last_error(PIE_EINVAL, "a lane number holds no call");
    N += lrows[size_t(l)];
    NP += int64_t(b->ws_pages[size_t(key[size_t(l)])].size());
  }
  {
    std::vector<int64_t> sorted(key);
    std::sort(sorted.begin(), sorted.end());
    if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end())
      return set_last_error(PIE_EINVAL, "a working set appears in two lanes of one batch");
  }
  *num_lanes = L;
  *num_rows = int32_t(std::min<int64_t>(N, INT32_MAX));
  *num_pages = NP;
  if (L > max_lanes || N > max_rows || NP > max_pages)
    return set_last_error(PIE_ENOSPACE, "the pass needs more lanes, rows or pages than given");
  if (N >= INT32_MAX || NP >= INT32_MAX) return set_last_error(PIE_ERANGE, "pass too large");
  if (!row_indptr || !positions || !kv_len || !page_indptr || !page_ids || !lane_keys)
    return set_last_error(PIE_EINVAL, "NULL output array");
  // lanes: rows at the working set's next free slots (position = slot), all
  // of the working set's pages, kv_len = frozen + rows
  row_indptr[0] = 0;
  page_indptr[0] = 0;
  for (int32_t l = 0; l < L; ++l) {
    const int64_t k = key[size_t(l)];
    const int32_t f = frozen[k];
    if (f < 0) return set_last_error(PIE_ERANGE, "negative frozen length");
    const std::vector<int32_t>& pg = b->ws_pages[size_t(k)];
    const int32_t r0 = row_indptr[l];
    row_indptr[l + 1] = r0 + int32_t(lrows[size_t(l)]);
    for (int32_t r = 0; r < int32_t(lrows[size_t(l)]); ++r) positions[r0 + r] = f + r;
    kv_len[l] = f + int32_t(lrows[size_t(l)]);
    std::memcpy(page_ids + page_indptr[l], pg.data(), pg.size() * sizeof(int32_t));
    page_indptr[l + 1] = page_indptr[l] + int32_t(pg.size());
    lane_keys[l] = k;
  }
  // each call's first row: its lane's rows in batch order
  std::vector<int32_t> cursor(row_indptr, row_indptr + L);
  for (int32_t i = 0; i < n; ++i) {
    first_row[i] = cursor[size_t(lanes[i])];
    cursor[size_t(lanes[i])] += int32_t(b->calls[size_t(calls[i])].rows);
  }
  return PIE_OK;
}

int pie_batcher_plan_forward(pie_batcher_t* b, const int64_t* calls, const int32_t* lanes, int32_t n,
                             const int32_t* frozen, int64_t num_keys, const pie_fwd_desc* desc,
                             int32_t num_pool_pages, void* dev_workspace, size_t ws_bytes,
                             void* stream, pie_fwd_plan_t** plan, int64_t* lane_keys,
                             int32_t* first_row, int32_t* kv_len, int32_t* num_lanes,
                             int32_t* num_rows) {
  if (!b || !plan || !lane_keys || !num_lanes || !num_rows || n < 1)
    return set_last_error(PIE_EINVAL, "NULL argument or an empty batch");
  *plan = nullptr;
  // sizes first (the capacity check of pie_batcher_forward_pass reports them)
  int32_t L = 0, N = 0;
  int64_t NP = 0;
  int rc = pie_batcher_forward_pass(b, calls, lanes, n, frozen, num_keys, 0, 0, 0, nullptr,
                                    nullptr, nullptr, nullptr, nullptr, nullptr, first_row, &L, &N,
                                    &NP);
  *num_lanes = L;
  *num_rows = N;
  if (rc != PIE_OK && rc != PIE_ENOSPACE) return rc;
  std::vector<int32_t>* v = b->pass_i32;
  v[0].resize(size_t(L) + 1);
  v[1].resize(std::max<size_t>(size_t(N), 1));
  v[2].resize(std::max<size_t>(size_t(L), 1));
  v[3].resize(size_t(L) + 1);
  v[4].resize(std::max<size_t>(size_t(NP), 1));
  v[5].assign(std::max<size_t>(size_t(L), 1), PIE_FOLD_ALL);
  rc = pie_batcher_forward_pass(b, calls, lanes, n, frozen, num_keys, L, N, NP, v[0].data(),
                                v[1].data(), v[2].data(), v[3].data(), v[4].data(), lane_keys,
                                first_row, &L, &N, &NP);
  if (rc != PIE_OK) return rc;
  if (kv_len) std::memcpy(kv_len, v[2].data(), size_t(L) * sizeof(int32_t));
  pie_fwd_meta m;
  std::memset(&m, 0, sizeof(m));
  m.num_lanes = L;
  m.num_rows = N;
  m.row_indptr = v[0].data();
  m.positions = v[1].data();
  m.slots = v[1].data();  // position = slot
  m.kv_len = v[2].data();
  m.page_indptr = v[3].data();
  m.page_ids = v[4].data();
  m.num_pool_pages = num_pool_pages;
  m.fold_mode = v[5].data();
  return pie_fwd_plan(desc, &m, dev_workspace, ws_bytes, stream, plan);
}

int pie_batcher_counts(const pie_batcher_t* b, int64_t* queued, int64_t* in_flight) {
  if (!b) return set_last_error(PIE_EINVAL, "batcher is NULL");
  if (queued) *queued = b->queued;
  if (in_flight) *in_flight = b->in_flight;
  return PIE_OK;
}

}  // extern "C"
