// seq.h -- what the head-side contexts (masked predictor, attentive-pool head) share around their
// launch sequences: the stream, CUDA-graph capture and replay keyed by the call's shape and
// pointers, per-launch event timing by kernel class, and the error-word check of a sync.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "internal.h"
#include "jepa.h"
#include "kernels.h"

namespace jepa {

struct SeqRunner {
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  // graph replay
  bool use_graph = false;
  cudaGraphExec_t gexec = nullptr;
  std::vector<uintptr_t> gkey;
  // profiling: events around each launch (eager launches only)
  bool profiling = false;
  std::vector<cudaEvent_t> ev;
  size_t ev_used = 0;
  struct Ev {
    int cls;
    size_t e0, e1;
    double flops, bytes;
  };
  std::vector<Ev> recs;
  std::vector<int> launches;
  std::vector<double> ms, flops, bytes;

  jepa_status init(int n_classes) {
    launches.assign(n_classes, 0);
    ms.assign(n_classes, 0.0);
    flops.assign(n_classes, 0.0);
    bytes.assign(n_classes, 0.0);
    CUDA_TRY(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    own_stream = true;
    return JEPA_OK;
  }

  void destroy() {
    if (stream) cudaStreamSynchronize(stream);
    if (gexec) cudaGraphExecDestroy(gexec);
    gexec = nullptr;
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    if (own_stream && stream) cudaStreamDestroy(stream);
    stream = nullptr;
  }

  jepa_status set_stream(void* s) {
    CUDA_TRY(cudaStreamSynchronize(stream));
    if (own_stream) cudaStreamDestroy(stream);
    stream = reinterpret_cast<cudaStream_t>(s);
    own_stream = false;
    if (gexec) {  // a graph recorded for another stream is dropped
      cudaGraphExecDestroy(gexec);
      gexec = nullptr;
    }
    return JEPA_OK;
  }

  // Runs `launch` (one kernel), bracketed by two events when profiling.
  template <class Fn>
  cudaError_t timed(int cls, double fl, double by, Fn&& launch) {
    if (!profiling) return launch();
    while (ev.size() < ev_used + 2) {
      cudaEvent_t e;
      const cudaError_t r = cudaEventCreate(&e);
      if (r != cudaSuccess) return r;
      ev.push_back(e);
    }
    const size_t e0 = ev_used++, e1 = ev_used++;
    cudaEventRecord(ev[e0], stream);
    const cudaError_t r = launch();
    cudaEventRecord(ev[e1], stream);
    recs.push_back({cls, e0, e1, fl, by});
    return r;
  }

  // Runs the launch sequence `seq` (returns jepa_status): eagerly, or from a CUDA graph captured on
  // the first call with this key and replayed while the key stays the same.
  template <class Fn>
  jepa_status run(const std::vector<uintptr_t>& key, Fn&& seq, const char* what) {
    if (!use_graph || profiling) return seq();
    if (!(gexec && key == gkey)) {
      if (gexec) {
        cudaGraphExecDestroy(gexec);
        gexec = nullptr;
      }
      cudaGraph_t graph = nullptr;
      CUDA_TRY(cudaStreamBeginCapture(stream, cudaStreamCaptureModeThreadLocal));
      const jepa_status st = seq();
      const cudaError_t e = cudaStreamEndCapture(stream, &graph);
      if (st != JEPA_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
      }
      if (e != cudaSuccess) return fail(JEPA_E_CUDA, "%s graph capture: %s", what, cudaGetErrorString(e));
      const cudaError_t ei = cudaGraphInstantiate(&gexec, graph, 0);
      cudaGraphDestroy(graph);
      if (ei != cudaSuccess) return fail(JEPA_E_CUDA, "%s graph instantiate: %s", what, cudaGetErrorString(ei));
      gkey = key;
    }
    CUDA_TRY(cudaGraphLaunch(gexec, stream));
    return JEPA_OK;
  }

  // Waits for the stream and reads (then clears) the device error word.
  jepa_status sync(int* err, const char* what) {
    CUDA_TRY(cudaStreamSynchronize(stream));
    int h = 0;
    CUDA_TRY(cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost));
    if (!h) return JEPA_OK;
    CUDA_TRY(cudaMemset(err, 0, sizeof(int)));
    if (h & kErrBadIds) return fail(JEPA_E_INVALID_ARG, "%s: an index argument was outside its range (replaced by 0)", what);
    return fail(JEPA_E_TIMEOUT, "%s: a device-side wait gave up (error word %d)", what, h);
  }

  // Folds the recorded events into per-class totals and reports them (as jepa_context_profile).
  jepa_status profile(const char* const* names, jepa_kernel_stat* out, int32_t max, int32_t* n_out, int32_t reset) {
    CUDA_TRY(cudaStreamSynchronize(stream));
    for (const auto& r : recs) {
      float t = 0.0f;
      CUDA_TRY(cudaEventElapsedTime(&t, ev[r.e0], ev[r.e1]));
      launches[r.cls] += 1;
      ms[r.cls] += t;
      flops[r.cls] += r.flops;
      bytes[r.cls] += r.bytes;
    }
    recs.clear();
    ev_used = 0;
    int n = 0;
    for (size_t k = 0; k < launches.size(); ++k) {
      if (!launches[k]) continue;
      if (n < max) {
        jepa_kernel_stat& st = out[n];
        memset(&st, 0, sizeof st);
        snprintf(st.name, sizeof st.name, "%s", names[k]);
        st.launches = launches[k];
        st.total_ms = (float)ms[k];
        st.flops = flops[k];
        st.bytes = bytes[k];
      }
      ++n;
    }
    *n_out = n;
    if (reset)
      for (size_t k = 0; k < launches.size(); ++k) {
        launches[k] = 0;
        ms[k] = flops[k] = bytes[k] = 0.0;
      }
    return JEPA_OK;
  }
};

// Launch mode of a sequence: programmatic dependent launches, except while profiling events are
// recorded between the kernels.
struct PdlScope {
  bool prev;
  explicit PdlScope(bool on) : prev(pdl_launches()) { pdl_launches() = on; }
  ~PdlScope() { pdl_launches() = prev; }
};

}  // namespace jepa
