// Residency manager: per-layer GPU slot pools fed from a complete, immutable
// page-locked host source, evicting by decayed access counts, by least recent
// use, or by least recent use outside a profile-pinned set.
//
// "Horizon RunMap -- Prévia Técnica", "03 / Arquitetura" (contract
// resident-qpacked-cache-v1, ADR 0009): the source in host RAM stays complete
// and is never rewritten; a copy lands in a GPU position while readers keep
// the previous generation; the new generation is published after the routed
// group's copies complete; an evicted slot is reused only after its readers
// retire; capacity is fixed before requests and init rejects a profile short
// of it; a failure before publish keeps the previous generation.
// "Desenvolvedor do Strata cria mapa ao vivo de 24 576 especialistas MoE em
// uma GTX 1070": eviction by an access counter whose old accesses lose weight.
// Horizon RunMap claims.json, experiment contract: canonical initial
// placement, evolving LRU. lucashiago.com.br "local" explainer, etapa 4: a
// profile measured beforehand pins the popular set; LRU adapts by itself.
// Prefetch (ADR 0009's spare positions): predicted misses are copied into
// free spare slots ahead of the step that needs them, without publishing;
// the step then takes them without a copy on its own path.
//
// Built with -ffp-contract=off: the count update c = c*decay; c = c + 1 is two
// IEEE double operations, with no fused multiply-add.
#include <algorithm>
#include <cstring>
#include <vector>

#include "common.h"
#include "kernels.h"

struct moe_residency {
  moe_residency_cfg cfg;
  const uint8_t* src = nullptr;
  uint8_t* pool = nullptr;
  int32_t* slot_of_dev = nullptr;
  cudaStream_t compute = nullptr, copy = nullptr;
  cudaEvent_t readers_done = nullptr, copies_done = nullptr;
  struct Layer {
    std::vector<double> counts;
    std::vector<int64_t> last_used;  // step of the last use, -1 never
    std::vector<char> pinned;        // never evicted (MOE_POLICY_PINNED)
    std::vector<int32_t> slot_of;  // expert -> physical slot, -1 absent
    std::vector<int32_t> free;     // free physical slots
    std::vector<int32_t> staged;   // expert -> spare slot holding a prefetched copy, -1 none
    moe_residency_stats st;
    int64_t steps = 0;
  };
  std::vector<Layer> layers;
  std::vector<moe_residency_event> trace;
  std::vector<moe_residency_op> ops;  // stream operations, when cfg.log_ops
  int64_t inject_countdown = -1;
  int physical = 0;
};

namespace {

// Every stream operation of the manager goes through these helpers: logged
// when the handle logs (cfg.log_ops), executed unless it is a dry run. The
// ordering decisions are therefore the same with and without a GPU.
enum { kCompute = 0, kCopy = 1 };
enum { kReadersDone = 0, kCopiesDone = 1 };  // event ids

void log_op(moe_residency* r, int kind, int stream, int event, int layer, int slot, int expert) {
  if (r->cfg.log_ops) r->ops.push_back({kind, stream, event, layer, slot, expert});
}
cudaEvent_t event_of(moe_residency* r, int ev) { return ev == kReadersDone ? r->readers_done : r->copies_done; }
cudaStream_t stream_of(moe_residency* r, int st) { return st == kCompute ? r->compute : r->copy; }

cudaError_t op_record(moe_residency* r, int ev, int st) {
  log_op(r, MOE_OP_RECORD, st, ev, -1, -1, -1);
  return r->cfg.dry_run ? cudaSuccess : cudaEventRecord(event_of(r, ev), stream_of(r, st));
}
cudaError_t op_wait(moe_residency* r, int st, int ev) {
  log_op(r, MOE_OP_WAIT, st, ev, -1, -1, -1);
  return r->cfg.dry_run ? cudaSuccess : cudaStreamWaitEvent(stream_of(r, st), event_of(r, ev), 0);
}
// Host -> device copy of `expert`'s block of `layer` into `slot`, on the copy stream.
cudaError_t op_copy(moe_residency* r, int layer, int slot, int expert) {
  log_op(r, MOE_OP_COPY, kCopy, -1, layer, slot, expert);
  if (r->cfg.dry_run) return cudaSuccess;
  const moe_residency_cfg& c = r->cfg;
  const uint8_t* src = r->src + ((size_t)layer * c.experts + expert) * c.block_bytes;
  uint8_t* dst = r->pool + ((size_t)layer * r->physical + slot) * c.block_bytes;
  return cudaMemcpyAsync(dst, src, c.block_bytes, cudaMemcpyHostToDevice, r->copy);
}

struct Miss {
  int32_t expert, slot, victim;
  bool staged;  // its block was copied by a prefetch: no copy in this step
};

int publish(moe_residency* r, int layer, const std::vector<std::pair<int32_t, int32_t>>& upd) {
  log_op(r, MOE_OP_PUBLISH, kCompute, -1, layer, -1, -1);
  if (r->cfg.dry_run) return MOE_OK;
  int32_t* table = r->slot_of_dev + (size_t)layer * r->cfg.experts;
  size_t i = 0;
  while (i < upd.size()) {
    moe::SlotUpdates u;
    u.n = 0;
    for (; i < upd.size() && u.n < moe::kMaxSlotUpdates; ++i, ++u.n) {
      u.expert[u.n] = upd[i].first;
      u.slot[u.n] = upd[i].second;
    }
    const int rc = moe::publish_slot_updates(table, u, r->compute);
    if (rc != MOE_OK) return rc;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_residency_create(const moe_residency_cfg* cfg, const void* host_src,
                         void* dev_pool, int32_t* dev_slot_of, void* compute,
                         void* copy, moe_residency** out) {
  moe::clear_error();
  if (!cfg || !out) return moe::fail(MOE_ERR_ARG, "moe_residency_create: NULL cfg/out");
  *out = nullptr;
  const moe_residency_cfg c = *cfg;
  if (c.layers < 1 || c.experts < 1 || c.spares < 0 || c.max_ids_per_step < 1 ||
      c.block_bytes == 0 || c.block_bytes % 16 || !(c.decay > 0.0 && c.decay <= 1.0))
    return moe::fail(MOE_ERR_ARG, "moe_residency_create: bad configuration");
  if (c.slots < 1 || c.slots > c.experts)
    return moe::fail(MOE_ERR_CAPACITY, "moe_residency_create: slots %d not in [1, E=%d]", c.slots, c.experts);
  if (std::min(c.max_ids_per_step, c.experts) > c.slots)
    return moe::fail(MOE_ERR_CAPACITY,
                     "moe_residency_create: a step may need %d distinct experts but only %d slots",
                     std::min(c.max_ids_per_step, c.experts), c.slots);
  if (c.slots + c.spares > 4096) return moe::fail(MOE_ERR_CAPACITY, "too many physical slots");
  if (c.policy < MOE_POLICY_DECAY || c.policy > MOE_POLICY_PINNED)
    return moe::fail(MOE_ERR_ARG, "moe_residency_create: unknown policy %d", c.policy);
  if (c.policy == MOE_POLICY_PINNED) {
    if (!c.profile || c.pinned < 0) return moe::fail(MOE_ERR_ARG, "moe_residency_create: pinned policy needs a profile");
    if (c.pinned > c.slots - std::min(c.max_ids_per_step, c.experts))
      return moe::fail(MOE_ERR_CAPACITY,
                       "moe_residency_create: %d pinned experts leave fewer than %d slots for a step's misses",
                       c.pinned, std::min(c.max_ids_per_step, c.experts));
  }
  if (!c.dry_run) {
    if (!host_src || !dev_pool || !dev_slot_of)
      return moe::fail(MOE_ERR_ARG, "moe_residency_create: NULL buffer");
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, host_src) != cudaSuccess || pa.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return moe::fail(MOE_ERR_ARG, "moe_residency_create: host_src must be page-locked host memory");
    }
  }
  moe_residency* r = new moe_residency();
  r->cfg = c;
  r->src = static_cast<const uint8_t*>(host_src);
  r->pool = static_cast<uint8_t*>(dev_pool);
  r->slot_of_dev = dev_slot_of;
  r->compute = static_cast<cudaStream_t>(compute);
  r->copy = static_cast<cudaStream_t>(copy);
  r->physical = c.slots + c.spares;
  r->layers.resize(c.layers);
  r->cfg.profile = nullptr;  // read here only
  for (int l = 0; l < c.layers; ++l) {
    auto& L = r->layers[l];
    L.counts.assign(c.experts, 0.0);
    L.last_used.assign(c.experts, -1);
    L.pinned.assign(c.experts, 0);
    L.slot_of.assign(c.experts, -1);
    L.staged.assign(c.experts, -1);
    if (c.policy == MOE_POLICY_PINNED) {
      // Top `pinned` experts by profile (ties: lower id), then the lowest
      // other ids; slots in ascending expert order.
      const double* prof = c.profile + (size_t)l * c.experts;
      std::vector<int32_t> order(c.experts);
      for (int e = 0; e < c.experts; ++e) order[e] = e;
      std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return prof[x] > prof[y]; });
      for (int i = 0; i < c.pinned; ++i) L.pinned[order[i]] = 1;
      std::vector<char> res(c.experts, 0);
      int n = 0;
      for (int e = 0; e < c.experts; ++e)
        if (L.pinned[e]) res[e] = 1, ++n;
      for (int e = 0; e < c.experts && n < c.slots; ++e)
        if (!res[e]) res[e] = 1, ++n;
      int s = 0;
      for (int e = 0; e < c.experts; ++e)
        if (res[e]) L.slot_of[e] = s++;
    } else {
      for (int e = 0; e < c.slots; ++e) L.slot_of[e] = e;
    }
    for (int s = c.slots; s < r->physical; ++s) L.free.push_back(s);
    std::memset(&L.st, 0, sizeof(L.st));
  }
  if (!c.dry_run) {
    cudaError_t e = cudaEventCreateWithFlags(&r->readers_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r->copies_done, cudaEventDisableTiming);
    // Initial placement: each resident expert's block into its slot
    // (canonical: expert e in slot e, e < C, one copy per layer).
    for (int l = 0; e == cudaSuccess && l < c.layers; ++l) {
      const uint8_t* s = r->src + (size_t)l * c.experts * c.block_bytes;
      uint8_t* d = r->pool + (size_t)l * r->physical * c.block_bytes;
      if (c.policy != MOE_POLICY_PINNED) {
        e = cudaMemcpy(d, s, (size_t)c.slots * c.block_bytes, cudaMemcpyHostToDevice);
      } else {
        for (int x = 0; e == cudaSuccess && x < c.experts; ++x) {
          const int32_t sl = r->layers[l].slot_of[x];
          if (sl >= 0)
            e = cudaMemcpy(d + (size_t)sl * c.block_bytes, s + (size_t)x * c.block_bytes, c.block_bytes,
                           cudaMemcpyHostToDevice);
        }
      }
    }
    if (e == cudaSuccess) {
      std::vector<int32_t> table((size_t)c.layers * c.experts);
      for (int l = 0; l < c.layers; ++l)
        std::memcpy(&table[(size_t)l * c.experts], r->layers[l].slot_of.data(), c.experts * 4);
      e = cudaMemcpy(dev_slot_of, table.data(), table.size() * 4, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
      moe_residency_destroy(r);
      return moe::fail(MOE_ERR_CUDA, "moe_residency_create: %s", cudaGetErrorString(e));
    }
  }
  *out = r;
  return MOE_OK;
}

int moe_residency_prepare(moe_residency* r, int layer, const int32_t* host_ids, int n) {
  moe::NvtxRange nvtx_range("moe_residency_prepare");
  moe::clear_error();
  if (!r) return moe::fail(MOE_ERR_ARG, "moe_residency_prepare: NULL handle");
  const moe_residency_cfg& c = r->cfg;
  if (layer < 0 || layer >= c.layers) return moe::fail(MOE_ERR_ARG, "layer %d out of range", layer);
  if (n < 0 || n > c.max_ids_per_step || (n > 0 && !host_ids))
    return moe::fail(MOE_ERR_ARG, "n = %d not in [0, max_ids_per_step = %d]", n, c.max_ids_per_step);
  for (int i = 0; i < n; ++i)
    if (host_ids[i] < 0 || host_ids[i] >= c.experts)
      return moe::fail(MOE_ERR_ARG, "id %d out of range [0, %d)", host_ids[i], c.experts);
  std::vector<int32_t> distinct(host_ids, host_ids + n);
  std::sort(distinct.begin(), distinct.end());
  distinct.erase(std::unique(distinct.begin(), distinct.end()), distinct.end());
  if ((int)distinct.size() > c.slots)
    return moe::fail(MOE_ERR_CAPACITY, "%zu distinct experts > %d slots", distinct.size(), c.slots);

  auto& L = r->layers[layer];
  // Plan on copies of the state; commit only after the step is enqueued.
  std::vector<double> counts = L.counts;
  for (int e = 0; e < c.experts; ++e) counts[e] = counts[e] * c.decay;
  for (int i = 0; i < n; ++i) counts[host_ids[i]] = counts[host_ids[i]] + 1.0;
  std::vector<int32_t> slot_of = L.slot_of;
  std::vector<int32_t> free_slots = L.free;
  std::vector<char> needed(c.experts, 0);
  for (int32_t e : distinct) needed[e] = 1;
  int n_resident = 0;
  for (int e = 0; e < c.experts; ++e) n_resident += slot_of[e] >= 0;
  std::vector<Miss> misses;
  std::vector<int32_t> retiring;
  int hits = 0;
  for (int32_t e : distinct) {
    if (slot_of[e] >= 0) {
      ++hits;
      continue;
    }
    int32_t victim = -1;
    if (n_resident == c.slots) {
      for (int v = 0; v < c.experts; ++v) {
        if (slot_of[v] < 0 || needed[v] || L.pinned[v]) continue;
        const bool better = c.policy == MOE_POLICY_DECAY ? counts[v] < counts[victim < 0 ? v : victim]
                                                          : L.last_used[v] < L.last_used[victim < 0 ? v : victim];
        if (victim < 0 || better) victim = v;  // ties keep the lower id
      }
      retiring.push_back(slot_of[victim]);
      slot_of[victim] = -1;
      --n_resident;
    }
    int32_t slot;
    const bool staged = L.staged[e] >= 0;
    if (staged) {
      slot = L.staged[e];  // prefetched: already in its spare slot
    } else if (!free_slots.empty()) {
      auto it = std::min_element(free_slots.begin(), free_slots.end());
      slot = *it;
      free_slots.erase(it);
    } else {
      slot = retiring.back();
      retiring.pop_back();
    }
    slot_of[e] = slot;
    ++n_resident;
    misses.push_back({e, slot, victim, staged});
  }
  for (int32_t s : retiring) free_slots.push_back(s);
  // Prefetched copies this step did not need return to the free spares.
  for (int e = 0; e < c.experts; ++e)
    if (L.staged[e] >= 0 && !needed[e]) free_slots.push_back(L.staged[e]);

  // Enqueue copies: the copy stream first waits for every reader enqueued so
  // far on the compute stream (this retires the victims' readers).
  int failed_at = -1;
  int rc = MOE_OK;
  if (!misses.empty()) {
    // Every reader of this step's victims is enqueued before this point. The
    // copy stream runs in order, so this wait also orders every later copy
    // into a slot freed here (a prefetch's) after those readers.
    cudaError_t e = op_record(r, kReadersDone, kCompute);
    if (e == cudaSuccess) e = op_wait(r, kCopy, kReadersDone);
    if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "residency ordering: %s", cudaGetErrorString(e));
  }
  for (size_t i = 0; i < misses.size(); ++i) {
    if (misses[i].staged) continue;
    if (r->inject_countdown == 0) {
      r->inject_countdown = -1;
      failed_at = (int)i;
      rc = moe::fail(MOE_ERR_INJECTED, "injected failure at copy %zu of layer %d", i, layer);
      break;
    }
    if (r->inject_countdown > 0) --r->inject_countdown;
    const Miss& m = misses[i];
    cudaError_t e = op_copy(r, layer, m.slot, m.expert);
    if (e != cudaSuccess) {
      failed_at = (int)i;
      rc = moe::fail(MOE_ERR_CUDA, "copy of expert %d: %s", m.expert, cudaGetErrorString(e));
      break;
    }
  }
  if (failed_at >= 0) {
    // Not published. Experts whose slots earlier copies of this step already
    // overwrote (in-place reuse of a victim's slot) are no longer valid:
    // mark them absent and publish only that removal.
    std::vector<std::pair<int32_t, int32_t>> removal;
    for (int i = 0; i < failed_at; ++i) {
      const Miss& m = misses[i];
      for (int v = 0; v < c.experts; ++v) {
        if (L.slot_of[v] == m.slot) {
          removal.push_back({v, -1});
          L.slot_of[v] = -1;
          L.free.push_back(m.slot);
        }
      }
    }
    if (!removal.empty()) {
      op_wait(r, kCompute, kReadersDone);
      publish(r, layer, removal);
    }
    return rc;
  }
  if (!misses.empty()) {
    std::vector<std::pair<int32_t, int32_t>> upd;
    for (const Miss& m : misses)
      if (m.victim >= 0) upd.push_back({m.victim, -1});
    for (const Miss& m : misses) upd.push_back({m.expert, m.slot});
    cudaError_t e = op_record(r, kCopiesDone, kCopy);
    if (e == cudaSuccess) e = op_wait(r, kCompute, kCopiesDone);
    if (e != cudaSuccess) return moe::fail(MOE_ERR_CUDA, "residency publish order: %s", cudaGetErrorString(e));
    const int prc = publish(r, layer, upd);
    if (prc != MOE_OK) return prc;
  }
  // Commit.
  for (const Miss& m : misses)
    r->trace.push_back({L.steps, layer, m.expert, m.slot, m.victim});
  for (int e = 0; e < c.experts; ++e) L.staged[e] = -1;
  L.counts.swap(counts);
  for (int32_t e : distinct) L.last_used[e] = L.steps;
  L.slot_of.swap(slot_of);
  L.free.swap(free_slots);
  L.st.steps += 1;
  L.st.hits += hits;
  L.st.misses += misses.size();
  for (const Miss& m : misses) {
    L.st.evictions += m.victim >= 0;
    L.st.prefetched += m.staged;
    if (!c.dry_run && !m.staged) {
      L.st.copies += 1;
      L.st.h2d_bytes += c.block_bytes;
    }
  }
  L.steps += 1;
  return MOE_OK;
}

int moe_residency_prefetch(moe_residency* r, int layer, const int32_t* host_ids, int n, int* staged_out) {
  moe::NvtxRange nvtx_range("moe_residency_prefetch");
  moe::clear_error();
  if (!r) return moe::fail(MOE_ERR_ARG, "moe_residency_prefetch: NULL handle");
  const moe_residency_cfg& c = r->cfg;
  if (layer < 0 || layer >= c.layers) return moe::fail(MOE_ERR_ARG, "layer %d out of range", layer);
  if (n < 0 || (n > 0 && !host_ids)) return moe::fail(MOE_ERR_ARG, "moe_residency_prefetch: bad id list");
  for (int i = 0; i < n; ++i)
    if (host_ids[i] < 0 || host_ids[i] >= c.experts)
      return moe::fail(MOE_ERR_ARG, "id %d out of range [0, %d)", host_ids[i], c.experts);
  auto& L = r->layers[layer];
  int staged = 0;
  // No wait: a free slot was either never read (a spare, or an unneeded
  // prefetched copy) or freed by a prepare() whose copy-stream wait already
  // follows every reader of its previous occupant.
  for (int i = 0; i < n && !L.free.empty(); ++i) {
    const int32_t e = host_ids[i];
    if (L.slot_of[e] >= 0 || L.staged[e] >= 0) continue;
    auto it = std::min_element(L.free.begin(), L.free.end());
    const int32_t slot = *it;
    if (r->inject_countdown == 0) {
      r->inject_countdown = -1;
      if (staged_out) *staged_out = staged;
      return moe::fail(MOE_ERR_INJECTED, "injected failure at a prefetch copy of layer %d", layer);
    }
    if (r->inject_countdown > 0) --r->inject_countdown;
    const cudaError_t err = op_copy(r, layer, slot, e);
    if (err != cudaSuccess) {
      if (staged_out) *staged_out = staged;
      return moe::fail(MOE_ERR_CUDA, "prefetch copy of expert %d: %s", e, cudaGetErrorString(err));
    }
    if (!c.dry_run) {
      L.st.copies += 1;
      L.st.h2d_bytes += c.block_bytes;
    }
    L.free.erase(it);
    L.staged[e] = slot;
    L.st.prefetch_copies += 1;
    ++staged;
  }
  if (staged_out) *staged_out = staged;
  return MOE_OK;
}

int moe_residency_get_stats(const moe_residency* r, int layer, moe_residency_stats* out) {
  moe::clear_error();
  if (!r || !out) return moe::fail(MOE_ERR_ARG, "NULL argument");
  std::memset(out, 0, sizeof(*out));
  if (layer >= r->cfg.layers || layer < -1) return moe::fail(MOE_ERR_ARG, "layer out of range");
  for (int l = 0; l < r->cfg.layers; ++l) {
    if (layer >= 0 && l != layer) continue;
    const auto& s = r->layers[l].st;
    out->steps += s.steps;
    out->hits += s.hits;
    out->misses += s.misses;
    out->evictions += s.evictions;
    out->copies += s.copies;
    out->h2d_bytes += s.h2d_bytes;
    out->prefetched += s.prefetched;
    out->prefetch_copies += s.prefetch_copies;
  }
  return MOE_OK;
}

int moe_residency_trace(const moe_residency* r, moe_residency_event* buf, size_t cap, size_t* n_out) {
  moe::clear_error();
  if (!r || !n_out || (cap && !buf)) return moe::fail(MOE_ERR_ARG, "NULL argument");
  *n_out = r->trace.size();
  const size_t n = std::min(cap, r->trace.size());
  if (n) std::memcpy(buf, r->trace.data(), n * sizeof(moe_residency_event));
  return MOE_OK;
}

int moe_residency_ops(const moe_residency* r, moe_residency_op* buf, size_t cap, size_t* n_out) {
  moe::clear_error();
  if (!r || !n_out || (cap && !buf)) return moe::fail(MOE_ERR_ARG, "NULL argument");
  *n_out = r->ops.size();
  const size_t n = std::min(cap, r->ops.size());
  if (n) std::memcpy(buf, r->ops.data(), n * sizeof(moe_residency_op));
  return MOE_OK;
}

int moe_residency_slot_table(const moe_residency* r, int layer, int32_t* host_out) {
  moe::clear_error();
  if (!r || !host_out || layer < 0 || layer >= r->cfg.layers) return moe::fail(MOE_ERR_ARG, "bad argument");
  std::memcpy(host_out, r->layers[layer].slot_of.data(), r->cfg.experts * sizeof(int32_t));
  return MOE_OK;
}

int moe_residency_counts(const moe_residency* r, int layer, double* host_out) {
  moe::clear_error();
  if (!r || !host_out || layer < 0 || layer >= r->cfg.layers) return moe::fail(MOE_ERR_ARG, "bad argument");
  std::memcpy(host_out, r->layers[layer].counts.data(), r->cfg.experts * sizeof(double));
  return MOE_OK;
}

int moe_residency_inject_copy_failure(moe_residency* r, int64_t nth_copy) {
  moe::clear_error();
  if (!r) return moe::fail(MOE_ERR_ARG, "NULL handle");
  r->inject_countdown = nth_copy < 0 ? -1 : nth_copy;
  return MOE_OK;
}

void moe_residency_destroy(moe_residency* r) {
  if (!r) return;
  if (!r->cfg.dry_run) {
    if (r->copy) cudaStreamSynchronize(r->copy);
    if (r->readers_done) cudaEventDestroy(r->readers_done);
    if (r->copies_done) cudaEventDestroy(r->copies_done);
  }
  delete r;
}

}  // extern "C"
