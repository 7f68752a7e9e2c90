// awq_search_host_layers: the scale search over a sequence of layers whose
// inputs and outputs live in host memory.
//
// A layer's search runs on the caller's stream; two library streams copy the
// next layer's X and weights in and the previous layer's results out at the
// same time.  Device inputs are double-buffered (two slots sized for the
// largest layer, from the library's pool); each search result is freed,
// stream-ordered, after its copy-out and after its host values were read.
// The call returns once every output is in the caller's host buffers.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "awq.h"
#include "awq_internal.h"

// Helpers shared with awq_api.cu (same thread-local error message and pool).
awq_status awq_internal_fail(awq_status st, const char* fmt, ...);
awq_status awq_internal_ok();
awq_status awq_internal_cuda_fail(cudaError_t e, const char* what);
awq_status awq_internal_check_cfg(const awq_qconfig* cfg);
bool awq_internal_k_fits(int64_t K, const awq_qconfig* cfg);
cudaError_t awq_internal_pool_alloc(void** p, size_t bytes, cudaStream_t st);

namespace {

// Host memory (pinned, or plain pageable) and not device memory: the host
// side may read and write it directly.
bool host_ptr(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return true;   // unknown to CUDA: ordinary host memory
  }
  return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

awq_status check_layer(const awq_host_layer& L, int li, const awq_qconfig* cfg) {
  if (L.X == nullptr || !host_ptr(L.X))
    return awq_internal_fail(AWQ_ERR_INVALID, "layers[%d].X must be host memory", li);
  if (L.T < 1 || (L.T > AWQ_MAX_STAT_TOKENS))
    return awq_internal_fail(AWQ_ERR_INVALID, "layers[%d].T=%lld (1..AWQ_MAX_STAT_TOKENS)", li,
                             static_cast<long long>(L.T));
  if (!awq_internal_k_fits(L.K, cfg) || (cfg->bits == 3 && L.K % 32) || L.K % 8)
    return awq_internal_fail(AWQ_ERR_INVALID,
                             "layers[%d].K=%lld does not fit bits=%d group_size=%d", li,
                             static_cast<long long>(L.K), cfg->bits, cfg->group_size);
  if (L.Ws == nullptr || L.n_w < 1 || L.n_w > AWQ_MAX_WEIGHTS)
    return awq_internal_fail(AWQ_ERR_INVALID, "layers[%d].n_w=%d (1..%d) with non-NULL Ws", li,
                             L.n_w, AWQ_MAX_WEIGHTS);
  if (L.codes == nullptr || L.scales == nullptr || L.zeros == nullptr || L.s == nullptr ||
      L.losses == nullptr || L.best == nullptr)
    return awq_internal_fail(AWQ_ERR_INVALID, "layers[%d] has a NULL output", li);
  for (int i = 0; i < L.n_w; ++i) {
    if (L.Ws[i].W == nullptr || !host_ptr(L.Ws[i].W) || L.Ws[i].N < 1)
      return awq_internal_fail(AWQ_ERR_INVALID,
                               "layers[%d].Ws[%d] must be host memory with N >= 1", li, i);
    if (L.codes[i] == nullptr || L.scales[i] == nullptr || L.zeros[i] == nullptr ||
        !host_ptr(L.codes[i]) || !host_ptr(L.scales[i]) || !host_ptr(L.zeros[i]))
      return awq_internal_fail(AWQ_ERR_INVALID,
                               "layers[%d]: codes/scales/zeros of weight %d must be host memory",
                               li, i);
  }
  if (!host_ptr(L.s) || !host_ptr(L.losses) || !host_ptr(L.best))
    return awq_internal_fail(AWQ_ERR_INVALID, "layers[%d]: s, losses, best must be host memory",
                             li);
  return AWQ_OK;
}

struct InFlight {
  int layer;
  awq_result* r;
  cudaEvent_t done;     // the search's work is complete
  cudaEvent_t copied;   // its outputs are in host memory
};

}  // namespace

extern "C" __attribute__((visibility("default"))) awq_status awq_search_host_layers(
    const awq_host_layer* layers, int n_layers, const awq_qconfig* cfg, void* stream) {
  awq::NvtxScope nvtx("awq_search_host_layers");
  if (n_layers < 0 || (n_layers > 0 && layers == nullptr))
    return awq_internal_fail(AWQ_ERR_INVALID, "n_layers=%d with layers %s", n_layers,
                             layers ? "set" : "NULL");
  awq_status st = awq_internal_check_cfg(cfg);
  if (st != AWQ_OK) return st;
  if (n_layers == 0) return awq_internal_ok();
  size_t x_max = 0, w_max = 0;
  for (int li = 0; li < n_layers; ++li) {
    if ((st = check_layer(layers[li], li, cfg)) != AWQ_OK) return st;
    const awq_host_layer& L = layers[li];
    size_t wb = 0;
    for (int i = 0; i < L.n_w; ++i) wb += static_cast<size_t>(L.Ws[i].N * L.K) * 2;
    x_max = std::max(x_max, static_cast<size_t>(L.T * L.K) * 2);
    w_max = std::max(w_max, wb);
  }
  x_max = (x_max + 255) & ~static_cast<size_t>(255);
  w_max = (w_max + 255) & ~static_cast<size_t>(255);

  cudaStream_t compute = static_cast<cudaStream_t>(stream);
  cudaStream_t s_in = nullptr, s_out = nullptr;
  void* slots = nullptr;
  std::vector<cudaEvent_t> events;
  std::vector<InFlight> pending;
  awq_status err = AWQ_OK;
  char err_msg[512] = "";

  auto new_event = [&](cudaEvent_t* ev) -> cudaError_t {
    const cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) events.push_back(*ev);
    return e;
  };
  // Record the first failure (status and message) and stop.
  auto record = [&](awq_status s) {
    if (err == AWQ_OK) {
      err = s;
      snprintf(err_msg, sizeof(err_msg), "%s", awq_last_error());
    }
  };
  auto cuda_step = [&](cudaError_t e, const char* what) -> bool {
    if (e == cudaSuccess) return true;
    record(awq_internal_cuda_fail(e, what));
    return false;
  };
  // Host values of a finished search, then its stream-ordered release once
  // its copy-out is done.
  auto retire = [&](const InFlight& f) -> bool {
    bool good = cuda_step(cudaEventSynchronize(f.done), "search completion");
    if (good) {
      const awq_status cs = awq_result_check(f.r);
      if (cs != AWQ_OK) {
        record(cs);
        good = false;
      } else {
        const awq_host_layer& L = layers[f.layer];
        memcpy(L.losses, awq_result_losses(f.r), sizeof(double) * cfg->n_grid);
        *L.best = awq_result_best_index(f.r);
      }
    }
    cudaStreamWaitEvent(compute, f.copied, 0);
    awq_free(f.r);
    return good;
  };

  bool ok = cuda_step(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking), "stream creation") &&
            cuda_step(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking), "stream creation");
  if (ok) {
    const cudaError_t e = awq_internal_pool_alloc(&slots, 2 * (x_max + w_max), compute);
    ok = cuda_step(e, "input slot allocation");
  }
  cudaEvent_t slots_ready = nullptr;
  ok = ok && cuda_step(new_event(&slots_ready), "event creation") &&
       cuda_step(cudaEventRecord(slots_ready, compute), "event record") &&
       cuda_step(cudaStreamWaitEvent(s_in, slots_ready, 0), "stream wait");
  cudaEvent_t slot_free[2] = {nullptr, nullptr};
  for (int li = 0; ok && li < n_layers; ++li) {
    const awq_host_layer& L = layers[li];
    const int k = li % 2;
    char* xs = static_cast<char*>(slots) + k * (x_max + w_max);
    char* ws = xs + x_max;
    // Inputs of layer li into slot k, once the search that last used it is done.
    if (slot_free[k] != nullptr && !cuda_step(cudaStreamWaitEvent(s_in, slot_free[k], 0),
                                              "stream wait"))
      break;
    if (!cuda_step(cudaMemcpyAsync(xs, L.X, static_cast<size_t>(L.T * L.K) * 2,
                                   cudaMemcpyHostToDevice, s_in),
                   "X copy"))
      break;
    awq_weight wd[AWQ_MAX_WEIGHTS];
    size_t off = 0;
    bool copies = true;
    for (int i = 0; i < L.n_w && copies; ++i) {
      const size_t b = static_cast<size_t>(L.Ws[i].N * L.K) * 2;
      wd[i].W = ws + off;
      wd[i].N = L.Ws[i].N;
      copies = cuda_step(cudaMemcpyAsync(ws + off, L.Ws[i].W, b, cudaMemcpyHostToDevice, s_in),
                         "W copy");
      off += (b + 15) & ~static_cast<size_t>(15);   // each weight 16-byte aligned
    }
    cudaEvent_t ready = nullptr, done = nullptr, copied = nullptr;
    if (!copies || !cuda_step(new_event(&ready), "event creation") ||
        !cuda_step(cudaEventRecord(ready, s_in), "event record") ||
        !cuda_step(cudaStreamWaitEvent(compute, ready, 0), "stream wait"))
      break;
    // The search, on the caller's stream.
    awq_result* r = nullptr;
    const awq_status ss = awq_search_layer(xs, L.T, L.K, nullptr, wd, L.n_w, cfg, compute, &r);
    if (ss != AWQ_OK) {
      record(ss);
      break;
    }
    if (!cuda_step(new_event(&done), "event creation") ||
        !cuda_step(cudaEventRecord(done, compute), "event record")) {
      pending.push_back({li, r, nullptr, nullptr});
      break;
    }
    slot_free[k] = done;
    // Its outputs out to the caller's host buffers.
    bool out_ok = cuda_step(cudaStreamWaitEvent(s_out, done, 0), "stream wait");
    const int64_t groups = cfg->group_size == -1 ? 1 : L.K / cfg->group_size;
    for (int i = 0; i < L.n_w && out_ok; ++i) {
      const int64_t n = L.Ws[i].N;
      out_ok = cuda_step(cudaMemcpyAsync(L.codes[i], awq_result_codes(r, i),
                                         static_cast<size_t>(awq_packed_words(n, L.K, cfg->bits)) * 4,
                                         cudaMemcpyDeviceToHost, s_out),
                         "codes copy") &&
               cuda_step(cudaMemcpyAsync(L.scales[i], awq_result_scales(r, i),
                                         static_cast<size_t>(n * groups) * 2,
                                         cudaMemcpyDeviceToHost, s_out),
                         "scales copy") &&
               cuda_step(cudaMemcpyAsync(L.zeros[i], awq_result_zeros(r, i),
                                         static_cast<size_t>(n * groups), cudaMemcpyDeviceToHost,
                                         s_out),
                         "zeros copy");
    }
    out_ok = out_ok &&
             cuda_step(cudaMemcpyAsync(L.s, awq_result_s(r), static_cast<size_t>(L.K) * 4,
                                       cudaMemcpyDeviceToHost, s_out),
                       "s copy") &&
             cuda_step(new_event(&copied), "event creation") &&
             cuda_step(cudaEventRecord(copied, s_out), "event record");
    pending.push_back({li, r, done, out_ok ? copied : nullptr});
    if (!out_ok) break;
    // Retire the previous layer while this one runs.
    if (pending.size() > 1) {
      const InFlight f = pending.front();
      pending.erase(pending.begin());
      if (!retire(f)) break;
    }
    ok = err == AWQ_OK;
  }
  if (err == AWQ_OK) {
    while (!pending.empty()) {
      const InFlight f = pending.front();
      pending.erase(pending.begin());
      if (!retire(f)) break;
    }
  }
  // Whatever happened: let every stream finish the work enqueued so far,
  // then release what is still held.
  if (s_in) cudaStreamSynchronize(s_in);
  if (s_out) cudaStreamSynchronize(s_out);
  cudaStreamSynchronize(compute);
  for (const InFlight& f : pending) awq_free(f.r);
  if (slots) cudaFreeAsync(slots, compute);
  cudaStreamSynchronize(compute);
  for (cudaEvent_t ev : events) cudaEventDestroy(ev);
  if (s_in) cudaStreamDestroy(s_in);
  if (s_out) cudaStreamDestroy(s_out);
  if (err != AWQ_OK) return awq_internal_fail(err, "%s", err_msg);
  return awq_internal_ok();
}
