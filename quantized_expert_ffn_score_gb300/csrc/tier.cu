// tier.cu -- experts beyond HBM: a heat-ranked set of expert records resident
// in HBM slots, the rest read in place from page-locked host (Grace) memory
// over NVLink-C2C by the same expert kernels, or absent.
//
// "Running a 2.78-Trillion-Parameter Model Across Two Desks", Act II: the
// experts of a model too large for one machine's fast memory are split into
// tiers ranked by how often they are used; Act III: an expert that is in no
// tier comes back as missing, never as a substitute.  WASTE README, "How it
// works": a bounded cache of expert records in fast memory in front of the
// slow store.  On a GB300 the slow store is the Grace memory next to the GPU:
// a record there is read over the C2C link by the kernels themselves (the
// record table simply points at it), and the hottest records are copied into
// HBM slots.
//
// The layer reads the tier's record table (moe_tier_desc.records) as its bank.
// moe_tier_observe adds a step's tokens-per-expert counts into a decayed heat
// on the device; moe_tier_rebalance reads the heat, ranks the experts and
// moves the hottest into the slots (moe_tier_plan is that ranking, pure host
// code), then rewrites the table.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void heat_kernel(float* heat, const int32_t* counts, int E, float decay) {
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x)
    heat[e] = decay * heat[e] + (float)counts[e];
}

}  // namespace
}  // namespace moe

struct moe_tier {
  moe_ctx* ctx;
  int device;
  moe_tier_desc desc;
  std::vector<const uint8_t*> host_dev;  // device-accessible address of each host copy (null: none)
  std::vector<int32_t> slot_of;          // expert -> slot, or -1
  std::vector<int32_t> expert_in;        // slot -> expert, or -1
  float* heat;                           // device [E]
  float* heat_host;                      // page-locked [E]
  const uint8_t** table_host;            // page-locked [E]: the table written to desc.records
};

namespace {

moe_status tier_ok(const moe_tier* t) {
  if (t == nullptr) return MOE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  return dev == t->device ? MOE_OK : MOE_ERR_INVALID_ARG;
}

// The table entry of expert e under the current residency.
const uint8_t* entry_of(const moe_tier* t, int e) {
  if (t->slot_of[e] >= 0) return t->desc.slots + (size_t)t->slot_of[e] * t->desc.slot_stride;
  return t->desc.direct_host ? t->host_dev[e] : nullptr;
}

moe_status write_table(moe_tier* t, cudaStream_t s) {
  for (int e = 0; e < t->desc.E; ++e) t->table_host[e] = entry_of(t, e);
  return cudaMemcpyAsync(const_cast<const uint8_t**>(t->desc.records), t->table_host, sizeof(void*) * t->desc.E,
                         cudaMemcpyHostToDevice, s) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// Moves the experts of `target` (all with a host copy, at most n_slots) into
// slots: evicted experts first point elsewhere in the table, then the copies
// run, then the table points at the new slots -- all on stream s.
moe_status apply_plan(moe_tier* t, const std::vector<int32_t>& new_slot_of, cudaStream_t s, int* n_moved) {
  const int E = t->desc.E;
  int moved = 0;
  for (int e = 0; e < E; ++e)  // an expert can only move into a slot from its host copy
    if (new_slot_of[e] >= 0 && new_slot_of[e] != t->slot_of[e] && t->desc.host_records[e] == nullptr)
      return MOE_ERR_INVALID_ARG;
  // 1. experts that leave their slot or move in: the table stops pointing at any slot that will be overwritten
  std::vector<int32_t> interim = t->slot_of;
  for (int e = 0; e < E; ++e)
    if (t->slot_of[e] >= 0 && new_slot_of[e] != t->slot_of[e]) interim[e] = -1;
  t->slot_of = interim;
  moe_status st = write_table(t, s);
  if (st != MOE_OK) return st;
  // 2. copies into the slots
  for (int e = 0; e < E; ++e) {
    if (new_slot_of[e] >= 0 && t->slot_of[e] != new_slot_of[e]) {
      const int sl = new_slot_of[e];
      if (cudaMemcpyAsync(t->desc.slots + (size_t)sl * t->desc.slot_stride, t->desc.host_records[e],
                          t->desc.record_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      ++moved;
    }
  }
  // 3. the final residency
  t->slot_of = new_slot_of;
  std::fill(t->expert_in.begin(), t->expert_in.end(), -1);
  for (int e = 0; e < E; ++e)
    if (t->slot_of[e] >= 0) t->expert_in[t->slot_of[e]] = e;
  if (n_moved) *n_moved = moved;
  return write_table(t, s);
}

}  // namespace

extern "C" {

int moe_tier_plan(int E, int n_slots, const float* heat, const uint8_t* has_host, const int32_t* slot_of,
                  int32_t* new_slot_of) {
  if (E <= 0 || n_slots < 0 || heat == nullptr || has_host == nullptr || slot_of == nullptr || new_slot_of == nullptr)
    return -1;
  // candidates: experts that can be resident (a host copy to load from, or already in a slot)
  std::vector<int> order;
  order.reserve(E);
  for (int e = 0; e < E; ++e)
    if (has_host[e] || (slot_of[e] >= 0 && slot_of[e] < n_slots)) order.push_back(e);
  // hottest first; equal heat: an expert already resident first (no copy), then the lower id
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    if (heat[a] != heat[b]) return heat[a] > heat[b];
    const bool ra = slot_of[a] >= 0, rb = slot_of[b] >= 0;
    if (ra != rb) return ra;
    return a < b;
  });
  const int keep = std::min<int>(n_slots, (int)order.size());
  std::vector<char> chosen(E, 0);
  for (int i = 0; i < keep; ++i) chosen[order[i]] = 1;
  // chosen experts already resident keep their slot; the others take the freed slots in ascending order
  std::vector<char> used(n_slots, 0);
  for (int e = 0; e < E; ++e) {
    new_slot_of[e] = -1;
    if (chosen[e] && slot_of[e] >= 0 && slot_of[e] < n_slots) {
      new_slot_of[e] = slot_of[e];
      used[slot_of[e]] = 1;
    }
  }
  int next = 0, moves = 0;
  for (int i = 0; i < keep; ++i) {
    const int e = order[i];
    if (new_slot_of[e] >= 0) continue;
    while (used[next]) ++next;
    new_slot_of[e] = next;
    used[next] = 1;
    ++moves;
  }
  return moves;
}

moe_status moe_tier_create(moe_ctx* ctx, const moe_tier_desc* d, moe_tier** out) {
  if (out == nullptr) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (ctx == nullptr || d == nullptr) return MOE_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (d->E <= 0 || d->E > moe::kMaxE * 2 || d->n_slots < 0 || d->n_slots > d->E) return MOE_ERR_INVALID_ARG;
  if (d->record_bytes == 0 || d->record_bytes % 16 || d->host_records == nullptr || d->records == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (d->n_slots > 0 && (d->slots == nullptr || d->slot_stride < d->record_bytes || d->slot_stride % 256 ||
                         (reinterpret_cast<uintptr_t>(d->slots) & 255u)))
    return MOE_ERR_INVALID_ARG;
  if (!(d->decay > 0.f && d->decay <= 1.f)) return MOE_ERR_INVALID_ARG;
  moe_tier* t = new (std::nothrow) moe_tier();
  if (t == nullptr) return MOE_ERR_CUDA;
  t->ctx = ctx;
  t->device = dev;
  t->desc = *d;
  t->host_dev.assign(d->E, nullptr);
  t->slot_of.assign(d->E, -1);
  t->expert_in.assign(d->n_slots, -1);
  t->heat = nullptr;
  t->heat_host = nullptr;
  t->table_host = nullptr;
  moe_status st = MOE_OK;
  for (int e = 0; e < d->E && st == MOE_OK; ++e) {
    const uint8_t* h = d->host_records[e];
    if (h == nullptr) continue;
    if (reinterpret_cast<uintptr_t>(h) & 255u) {
      st = MOE_ERR_INVALID_ARG;  // the kernels read records with aligned bulk copies
      break;
    }
    // page-locked memory only: where the GPU can also reach pageable memory
    // through the host's page tables, the device-pointer query alone would
    // accept pageable memory too
    cudaPointerAttributes pa;
    void* p = nullptr;
    if (cudaPointerGetAttributes(&pa, h) != cudaSuccess || pa.type != cudaMemoryTypeHost ||
        cudaHostGetDevicePointer(&p, const_cast<uint8_t*>(h), 0) != cudaSuccess) {
      cudaGetLastError();
      st = MOE_ERR_INVALID_ARG;  // not page-locked, mapped host memory
      break;
    }
    t->host_dev[e] = static_cast<const uint8_t*>(p);
  }
  if (st == MOE_OK &&
      (cudaMalloc(&t->heat, sizeof(float) * d->E) != cudaSuccess ||
       cudaMemset(t->heat, 0, sizeof(float) * d->E) != cudaSuccess ||
       cudaMallocHost(&t->heat_host, sizeof(float) * d->E) != cudaSuccess ||
       cudaMallocHost(reinterpret_cast<void**>(&t->table_host), sizeof(void*) * d->E) != cudaSuccess))
    st = MOE_ERR_CUDA;
  if (st == MOE_OK) {  // nothing resident yet: the table points at the host copies (or nowhere)
    st = write_table(t, 0);
    if (st == MOE_OK && cudaStreamSynchronize(0) != cudaSuccess) st = MOE_ERR_CUDA;
  }
  if (st != MOE_OK) {
    moe_tier_destroy(t);
    return st;
  }
  *out = t;
  return MOE_OK;
}

void moe_tier_destroy(moe_tier* t) {
  if (t == nullptr) return;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(t->device);
  if (t->heat) cudaFree(t->heat);
  if (t->heat_host) cudaFreeHost(t->heat_host);
  if (t->table_host) cudaFreeHost(t->table_host);
  cudaSetDevice(prev);
  delete t;
}

moe_status moe_tier_observe(moe_tier* t, const int32_t* counts, cudaStream_t stream) {
  moe_status st = tier_ok(t);
  if (st != MOE_OK) return st;
  if (counts == nullptr) return MOE_ERR_INVALID_ARG;
  moe::ProfScope prof_scope(t->ctx);
  const int blocks = (t->desc.E + 255) / 256;
  return moe::launch("tier_heat", moe::heat_kernel, dim3(blocks), dim3(256), 0, stream, false, t->heat, counts,
                     t->desc.E, t->desc.decay) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_tier_rebalance(moe_tier* t, cudaStream_t stream, int* n_moved) {
  moe_status st = tier_ok(t);
  if (st != MOE_OK) return st;
  if (n_moved) *n_moved = 0;
  if (cudaMemcpyAsync(t->heat_host, t->heat, sizeof(float) * t->desc.E, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  std::vector<uint8_t> has(t->desc.E);
  for (int e = 0; e < t->desc.E; ++e) has[e] = t->desc.host_records[e] != nullptr;
  std::vector<int32_t> plan(t->desc.E);
  if (moe_tier_plan(t->desc.E, t->desc.n_slots, t->heat_host, has.data(), t->slot_of.data(), plan.data()) < 0)
    return MOE_ERR_INVALID_ARG;
  return apply_plan(t, plan, stream, n_moved);
}

moe_status moe_tier_pin(moe_tier* t, const int32_t* experts, int n, cudaStream_t stream) {
  moe_status st = tier_ok(t);
  if (st != MOE_OK) return st;
  if (n < 0 || n > t->desc.n_slots || (n > 0 && experts == nullptr)) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  // the listed experts rank above every other expert, in list order; then the heat
  std::vector<float> score(t->desc.E, -1.f);
  std::vector<uint8_t> has(t->desc.E);
  for (int e = 0; e < t->desc.E; ++e) has[e] = t->desc.host_records[e] != nullptr;
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= t->desc.E || !(has[e] || t->slot_of[e] >= 0)) return MOE_ERR_INVALID_ARG;
    score[e] = (float)(n - i);
  }
  std::vector<int32_t> plan(t->desc.E);
  std::vector<int32_t> cur = t->slot_of;
  if (moe_tier_plan(t->desc.E, n, score.data(), has.data(), cur.data(), plan.data()) < 0) return MOE_ERR_INVALID_ARG;
  // experts beyond the pinned ones keep their slots when those slots are still free
  std::vector<char> used(t->desc.n_slots, 0);
  for (int e = 0; e < t->desc.E; ++e)
    if (plan[e] >= 0) used[plan[e]] = 1;
  for (int e = 0; e < t->desc.E; ++e)
    if (plan[e] < 0 && cur[e] >= 0 && !used[cur[e]]) {
      plan[e] = cur[e];
      used[cur[e]] = 1;
    }
  return apply_plan(t, plan, stream, nullptr);
}

moe_status moe_tier_residency(const moe_tier* t, int32_t* slot_of_expert, float* heat) {
  moe_status st = tier_ok(t);
  if (st != MOE_OK) return st;
  if (slot_of_expert) std::memcpy(slot_of_expert, t->slot_of.data(), sizeof(int32_t) * t->desc.E);
  if (heat && cudaMemcpy(heat, t->heat, sizeof(float) * t->desc.E, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // extern "C"
