// Single-GPU tile-task executor.
//
// The NNTile pages describe training as a sequential task flow: layers submit
// tasks in program order, each task declares the tiles it reads and writes,
// and a runtime infers the dependencies and runs ready tasks on any unit while
// moving tiles asynchronously (review page "What carries the argument"; first
// page, abstract). On one GB300 the plan is static, so it is built once:
//
//   * dependency inference over tile accesses (read-after-write,
//     write-after-read, write-after-write) when the program is finalised;
//   * a stream schedule: a task continues the stream of the dependency it
//     directly follows, independent tasks spread over the other streams, and
//     only the cross-stream edges that are not already implied by earlier
//     waits become cudaStreamWaitEvent calls;
//   * run = fork from the caller's stream, launch every task in order on its
//     stream, join back (optionally captured once into a CUDA graph and then
//     replayed with one launch).
#pragma once
#include <cuda_runtime.h>

#include <functional>
#include <string>
#include <vector>

#include "nnt.h"

namespace nnt {

enum Access : int { ACC_R = 1, ACC_W = 2, ACC_RW = 3 };

struct TileUse {
  int64_t tile;
  int mode;
};

struct Task {
  int type = 0;
  std::vector<TileUse> uses;
  std::function<nnt_status(cudaStream_t)> fn;
  double flops = 0, bytes = 0;
  int copy_engine = 0;  // 1: host<->device copy task, scheduled on the copy stream
  int kernels = 1;      // kernel launches the task makes
  int stream_hint = -1; // >= 0: run on this compute stream (side work kept off the main chain)
  // schedule (finalize)
  int stream = 0;
  std::vector<int> waits;
  bool record = false;
};

class Program {
 public:
  int add(Task t);
  // Infer dependencies and assign streams (n_streams compute streams, plus one
  // copy stream when any task is a copy task).
  void finalize(int n_streams);
  size_t size() const { return tasks_.size(); }
  const std::vector<Task>& tasks() const { return tasks_; }
  int n_edges() const { return n_edges_; }
  int n_streams_used() const { return n_streams_used_; }
  int64_t kernels() const {
    int64_t k = 0;
    for (const Task& t : tasks_) k += t.kernels;
    return k;
  }
  const std::vector<std::vector<int>>& deps() const { return deps_; }

  std::vector<Task> tasks_;
  std::vector<std::vector<int>> deps_;
  int n_streams_ = 1;
  int n_edges_ = 0;
  int n_streams_used_ = 1;
};

// Stream/event resources shared by every program of a model.
class Executor {
 public:
  ~Executor();
  nnt_status init(cudaStream_t main, int n_streams, bool need_copy_stream, bool trace,
                  int n_types);
  // Launch the program. `graph_slot` >= 0 captures it on first use and replays
  // the captured graph afterwards.
  nnt_status run(Program& p, int graph_slot);
  // After the stream is synchronised: fold the last traced run into per-type
  // totals (no-op unless tracing).
  nnt_status collect_trace(const Program& p);
  void reset_trace();
  void set_trace(bool on) { trace_ = on; }
  void drop_graphs() {
    for (auto& g : graphs_)
      if (g) {
        cudaGraphExecDestroy(g);
        g = nullptr;
      }
  }

  cudaStream_t main_ = nullptr;
  std::vector<cudaStream_t> streams_;  // [0] = main, then side streams, then copy stream
  int n_compute_ = 1;
  bool trace_ = false;
  std::vector<cudaEvent_t> task_events_;
  std::vector<cudaEvent_t> t0_, t1_;
  std::vector<cudaEvent_t> fork_join_;
  std::vector<cudaGraphExec_t> graphs_;
  int n_types_ = 0;
  std::vector<int64_t> type_launches_;
  std::vector<double> type_ms_, type_flops_, type_bytes_;

 private:
  nnt_status launch_all(Program& p, bool traced, bool capturing);
  nnt_status ensure_events(size_t n);
};

}  // namespace nnt
