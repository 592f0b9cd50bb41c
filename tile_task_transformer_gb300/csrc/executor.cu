// Tile-task executor: dependency inference, stream schedule, launch, trace.
#include <algorithm>
#include <unordered_map>

#include "common.cuh"
#include "executor.h"

namespace nnt {

int Program::add(Task t) {
  tasks_.push_back(std::move(t));
  return (int)tasks_.size() - 1;
}

void Program::finalize(int n_streams) {
  n_streams_ = std::max(1, n_streams);
  const size_t n = tasks_.size();
  deps_.assign(n, {});
  struct TileState {
    int writer = -1;
    std::vector<int> readers;
  };
  std::unordered_map<int64_t, TileState> state;
  std::unordered_map<int64_t, int> modes;
  for (size_t i = 0; i < n; ++i) {
    modes.clear();
    for (const TileUse& u : tasks_[i].uses) modes[u.tile] |= u.mode;
    std::vector<int>& d = deps_[i];
    for (const auto& kv : modes) {
      TileState& s = state[kv.first];
      if (s.writer >= 0) d.push_back(s.writer);              // RAW, WAW
      if (kv.second & ACC_W) d.insert(d.end(), s.readers.begin(), s.readers.end());  // WAR
    }
    for (const auto& kv : modes) {
      TileState& s = state[kv.first];
      if (kv.second & ACC_W) {
        s.writer = (int)i;
        s.readers.clear();
      } else {
        s.readers.push_back((int)i);
      }
    }
    std::sort(d.begin(), d.end());
    d.erase(std::unique(d.begin(), d.end()), d.end());
    d.erase(std::remove(d.begin(), d.end(), (int)i), d.end());
  }

  bool has_copy = false;
  for (const Task& t : tasks_) has_copy |= t.copy_engine != 0;
  const int ns = n_streams_ + (has_copy ? 1 : 0);
  const int copy_stream = n_streams_;
  for (Task& t : tasks_) t.record = false;
  std::vector<int> last_on(ns, -1);
  std::vector<std::vector<int>> frontier(n, std::vector<int>(ns, -1));
  n_edges_ = 0;
  std::vector<char> used(ns, 0);
  for (size_t i = 0; i < n; ++i) {
    Task& t = tasks_[i];
    int s;
    if (t.copy_engine) {
      s = copy_stream;
    } else if (t.stream_hint >= 0) {
      s = std::min(t.stream_hint, n_streams_ - 1);
    } else {
      // continue the stream whose latest task is one of our dependencies
      s = -1;
      for (int c = 0; c < n_streams_; ++c) {
        if (last_on[c] < 0) continue;
        if (std::binary_search(deps_[i].begin(), deps_[i].end(), last_on[c]) &&
            (s < 0 || last_on[c] > last_on[s]))
          s = c;
      }
      if (s < 0) {  // least recently used compute stream
        s = 0;
        for (int c = 1; c < n_streams_; ++c)
          if (last_on[c] < last_on[s]) s = c;
      }
    }
    t.stream = s;
    used[s] = 1;
    std::vector<int> F(ns, -1);
    if (last_on[s] >= 0) {
      F = frontier[last_on[s]];
      F[s] = std::max(F[s], last_on[s]);
    }
    t.waits.clear();
    for (auto it = deps_[i].rbegin(); it != deps_[i].rend(); ++it) {
      const int dep = *it;
      const int sd = tasks_[dep].stream;
      if (dep <= F[sd]) continue;  // already implied
      t.waits.push_back(dep);
      tasks_[dep].record = true;
      ++n_edges_;
      for (int c = 0; c < ns; ++c) F[c] = std::max(F[c], frontier[dep][c]);
      F[sd] = std::max(F[sd], dep);
    }
    frontier[i] = F;
    last_on[s] = (int)i;
  }
  n_streams_used_ = 0;
  for (char u : used) n_streams_used_ += u;
}

}  // namespace nnt

extern "C" nnt_status nnt_plan_schedule(int32_t n_tasks, const int64_t* use_off,
                                        const int64_t* use_tile, const int32_t* use_mode,
                                        const int32_t* copy_task, const int32_t* stream_hint,
                                        int32_t n_streams, int32_t* stream_out, int64_t* dep_off,
                                        int32_t* dep_task, int64_t dep_cap, int64_t* wait_off,
                                        int32_t* wait_task, int64_t wait_cap) {
  using namespace nnt;
  NNT_CHECK_ARG(n_tasks >= 0 && n_streams >= 1, "plan_schedule: n_tasks %d, n_streams %d", n_tasks,
                n_streams);
  NNT_CHECK_ARG(use_off && stream_out && dep_off && wait_off, "plan_schedule: NULL array");
  NNT_CHECK_ARG(use_off[0] == 0, "plan_schedule: use_off[0] must be 0");
  for (int32_t i = 0; i < n_tasks; ++i)
    NNT_CHECK_ARG(use_off[i + 1] >= use_off[i], "plan_schedule: use_off decreases at task %d", i);
  const int64_t n_uses = use_off[n_tasks];
  NNT_CHECK_ARG(n_uses == 0 || (use_tile && use_mode), "plan_schedule: NULL tile or mode array");
  for (int64_t u = 0; u < n_uses; ++u)
    NNT_CHECK_ARG(use_mode[u] >= 1 && use_mode[u] <= 3, "plan_schedule: mode %d at use %lld",
                  use_mode[u], (long long)u);
  Program p;
  for (int32_t i = 0; i < n_tasks; ++i) {
    Task t;
    for (int64_t u = use_off[i]; u < use_off[i + 1]; ++u) t.uses.push_back({use_tile[u], use_mode[u]});
    t.copy_engine = copy_task ? (copy_task[i] != 0) : 0;
    t.stream_hint = stream_hint ? std::max(-1, stream_hint[i]) : -1;
    p.add(std::move(t));
  }
  p.finalize(n_streams);
  dep_off[0] = 0;
  wait_off[0] = 0;
  for (int32_t i = 0; i < n_tasks; ++i) {
    dep_off[i + 1] = dep_off[i] + (int64_t)p.deps()[i].size();
    wait_off[i + 1] = wait_off[i] + (int64_t)p.tasks()[i].waits.size();
  }
  NNT_CHECK_ARG(dep_off[n_tasks] <= dep_cap && wait_off[n_tasks] <= wait_cap,
                "plan_schedule: %lld dependencies and %lld waits do not fit capacities %lld, %lld",
                (long long)dep_off[n_tasks], (long long)wait_off[n_tasks], (long long)dep_cap,
                (long long)wait_cap);
  NNT_CHECK_ARG((dep_off[n_tasks] == 0 || dep_task) && (wait_off[n_tasks] == 0 || wait_task),
                "plan_schedule: NULL dependency or wait array");
  for (int32_t i = 0; i < n_tasks; ++i) {
    stream_out[i] = p.tasks()[i].stream;
    std::copy(p.deps()[i].begin(), p.deps()[i].end(), dep_task + dep_off[i]);
    std::copy(p.tasks()[i].waits.begin(), p.tasks()[i].waits.end(), wait_task + wait_off[i]);
  }
  return NNT_OK;
}

namespace nnt {

Executor::~Executor() {
  for (auto g : graphs_)
    if (g) cudaGraphExecDestroy(g);
  for (auto e : task_events_) cudaEventDestroy(e);
  for (auto e : t0_) cudaEventDestroy(e);
  for (auto e : t1_) cudaEventDestroy(e);
  for (auto e : fork_join_) cudaEventDestroy(e);
  for (size_t i = 1; i < streams_.size(); ++i) cudaStreamDestroy(streams_[i]);
}

nnt_status Executor::init(cudaStream_t main, int n_streams, bool need_copy_stream, bool trace,
                          int n_types) {
  main_ = main;
  n_compute_ = std::max(1, n_streams);
  trace_ = trace;
  streams_.assign(1, main);
  const int total = n_compute_ + (need_copy_stream ? 1 : 0);
  for (int i = 1; i < total; ++i) {
    cudaStream_t s;
    NNT_CUDA_TRY(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    streams_.push_back(s);
  }
  if (need_copy_stream && total == 1) {
    cudaStream_t s;
    NNT_CUDA_TRY(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    streams_.push_back(s);
  }
  fork_join_.resize(streams_.size() + 1);
  for (auto& e : fork_join_) NNT_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
  graphs_.assign(8, nullptr);
  n_types_ = n_types;
  reset_trace();
  return NNT_OK;
}

void Executor::reset_trace() {
  type_launches_.assign(n_types_, 0);
  type_ms_.assign(n_types_, 0.0);
  type_flops_.assign(n_types_, 0.0);
  type_bytes_.assign(n_types_, 0.0);
}

nnt_status Executor::ensure_events(size_t n) {
  while (task_events_.size() < n) {
    cudaEvent_t e;
    NNT_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    task_events_.push_back(e);
  }
  if (trace_) {
    while (t0_.size() < n) {
      cudaEvent_t a, b;
      NNT_CUDA_TRY(cudaEventCreate(&a));
      NNT_CUDA_TRY(cudaEventCreate(&b));
      t0_.push_back(a);
      t1_.push_back(b);
    }
  }
  return NNT_OK;
}

nnt_status Executor::launch_all(Program& p, bool traced, bool capturing) {
  NNT_TRY(ensure_events(p.size()));
  const int ns = (int)streams_.size();
  NNT_CUDA_TRY(cudaEventRecord(fork_join_[0], main_));
  for (int s = 1; s < ns; ++s) NNT_CUDA_TRY(cudaStreamWaitEvent(streams_[s], fork_join_[0], 0));
  for (size_t i = 0; i < p.tasks_.size(); ++i) {
    Task& t = p.tasks_[i];
    cudaStream_t s = streams_[std::min(t.stream, ns - 1)];
    for (int w : t.waits) NNT_CUDA_TRY(cudaStreamWaitEvent(s, task_events_[w], 0));
    // inside a capture, timing events become external event-record nodes
    if (traced)
      NNT_CUDA_TRY(capturing ? cudaEventRecordWithFlags(t0_[i], s, cudaEventRecordExternal)
                             : cudaEventRecord(t0_[i], s));
    NNT_TRY(t.fn(s));
    if (traced)
      NNT_CUDA_TRY(capturing ? cudaEventRecordWithFlags(t1_[i], s, cudaEventRecordExternal)
                             : cudaEventRecord(t1_[i], s));
    if (t.record) NNT_CUDA_TRY(cudaEventRecord(task_events_[i], s));
  }
  for (int s = 1; s < ns; ++s) {
    NNT_CUDA_TRY(cudaEventRecord(fork_join_[s], streams_[s]));
    NNT_CUDA_TRY(cudaStreamWaitEvent(main_, fork_join_[s], 0));
  }
  return NNT_OK;
}

nnt_status Executor::run(Program& p, int graph_slot) {
  if (graph_slot < 0) return launch_all(p, trace_, false);
  // traced programs get their own graphs (with timing-event nodes) in slot + 4
  if (trace_) {
    NNT_TRY(ensure_events(p.size()));
    graph_slot += 4;
  }
  if ((size_t)graph_slot >= graphs_.size()) graphs_.resize(graph_slot + 1, nullptr);
  if (!graphs_[graph_slot]) {
    cudaGraph_t g = nullptr;
    NNT_CUDA_TRY(cudaStreamBeginCapture(main_, cudaStreamCaptureModeThreadLocal));
    nnt_status st = launch_all(p, trace_, true);
    cudaError_t e = cudaStreamEndCapture(main_, &g);
    if (st != NNT_OK) {
      if (g) cudaGraphDestroy(g);
      return st;
    }
    if (e != cudaSuccess) {
      set_thread_error("graph capture failed: %s", cudaGetErrorString(e));
      return NNT_ERR_CUDA;
    }
    cudaGraphExec_t ge = nullptr;
    e = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      set_thread_error("graph instantiate failed: %s", cudaGetErrorString(e));
      return NNT_ERR_CUDA;
    }
    graphs_[graph_slot] = ge;
  }
  NNT_CUDA_TRY(cudaGraphLaunch(graphs_[graph_slot], main_));
  return NNT_OK;
}

nnt_status Executor::collect_trace(const Program& p) {
  if (!trace_) return NNT_OK;
  for (size_t i = 0; i < p.tasks_.size(); ++i) {
    const Task& t = p.tasks_[i];
    float ms = 0.f;
    NNT_CUDA_TRY(cudaEventElapsedTime(&ms, t0_[i], t1_[i]));
    if (t.type >= 0 && t.type < n_types_) {
      type_launches_[t.type] += 1;
      type_ms_[t.type] += ms;
      type_flops_[t.type] += t.flops;
      type_bytes_[t.type] += t.bytes;
    }
  }
  return NNT_OK;
}

}  // namespace nnt
