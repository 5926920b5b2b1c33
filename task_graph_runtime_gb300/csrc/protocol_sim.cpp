// CPU model of the persistent runtime's protocol, on a built graph's own
// device encoding: one std::thread per worker CTA leader and per scheduler
// warp, std::atomic event counters with the epoch rule, per-worker AOT
// queues in linear order (the 64-byte AOT records, including the cached
// fan-out), JIT dispatch through scheduler rings and per-worker rings, and
// empty tasks run inline by the activating trigger -- the same decisions
// the kernel's worker_consumers / scheduler_role / trigger take (MPK: A
// Compiler and Runtime for Mega-Kernelizing Tensor Programs, §2 Q2 runtime
// and Figure 8, AOT vs JIT).  Task bodies are replaced by random delays.
// Which worker a JIT task goes to does not change the protocol; the model
// deals JIT tasks round-robin (the kernel deals attention chunks by cost).
//
// Checked for every executed task: it runs exactly once per step, and every
// task that triggers the event it waits on has finished in the same step
// before it starts (producer before consumer).  A step that does not finish
// within the time limit is reported as deadlocked.
#include <atomic>
#include <chrono>
#include <cstring>
#include <memory>
#include <random>
#include <thread>
#include <vector>

#include "device_abi.h"
#include "graph_state.h"
#include "mpk.h"

namespace {

using namespace mpk;
using Clock = std::chrono::steady_clock;

struct SimRing {
  std::atomic<uint32_t> head{0}, tail{0};
  std::vector<std::atomic<uint64_t>> slots;
  explicit SimRing(uint32_t cap) : slots(cap) {
    for (auto& s : slots) s.store(0, std::memory_order_relaxed);
  }
};

struct Sim {
  const mpk_graph* g;
  int W, S, nT, nE;
  uint32_t epoch = 0;
  std::vector<std::atomic<uint32_t>> counters;
  std::vector<std::unique_ptr<SimRing>> jit, sched;
  std::vector<std::atomic<uint32_t>> done_epoch;   // per task: last step run
  std::vector<std::atomic<int32_t>> runs;          // per task: runs this step
  std::vector<std::vector<int32_t>> producers;     // per event: its triggers
  std::atomic<int64_t> tasks_run{0}, order_violations{0};
  std::atomic<bool> abort{false};
  Clock::time_point deadline;
  int max_delay_us;

  Sim(const mpk_graph* gr, int delay_us)
      : g(gr),
        W(gr->bg.cfg.num_workers),
        S(gr->num_sched_sms * gr->sched_warps_per_sm),
        nT((int)gr->h_tasks.size()),
        nE((int)gr->h_events.size()),
        counters(nE),
        done_epoch(nT),
        runs(nT),
        producers(nE),
        max_delay_us(delay_us) {
    for (auto& c : counters) c.store(0);
    for (auto& d : done_epoch) d.store(0);
    for (int w = 0; w < W; ++w)
      jit.emplace_back(std::make_unique<SimRing>(mpk_detail::kJitCap));
    for (int s = 0; s < S; ++s)
      sched.emplace_back(std::make_unique<SimRing>(mpk_detail::kSchedCap));
    for (int t = 0; t < nT; ++t)
      if (g->h_tasks[t].trig >= 0 && g->h_tasks[t].trig < nE)
        producers[g->h_tasks[t].trig].push_back(t);
  }

  bool timed_out() {
    if (abort.load(std::memory_order_relaxed)) return true;
    if (Clock::now() > deadline) {
      abort.store(true);
      return true;
    }
    return false;
  }

  bool event_done(int e, uint32_t count) {
    return (int32_t)(counters[e].load(std::memory_order_acquire) -
                     epoch * count) >= 0;
  }

  // ring push (multi-producer) and pop (single consumer), ticketed slots
  bool push(SimRing& r, uint32_t v) {
    const uint32_t pos = r.tail.fetch_add(1u);
    const uint32_t cap = (uint32_t)r.slots.size();
    while (pos - r.head.load(std::memory_order_acquire) >= cap) {
      if (timed_out()) return false;
      std::this_thread::yield();
    }
    r.slots[pos % cap].store(((uint64_t)(pos + 1u) << 32) | v,
                             std::memory_order_release);
    return true;
  }
  bool try_pop(SimRing& r, uint32_t& head, uint32_t& v) {
    const uint32_t cap = (uint32_t)r.slots.size();
    const uint64_t x = r.slots[head % cap].load(std::memory_order_acquire);
    if ((uint32_t)(x >> 32) != head + 1u) return false;
    v = (uint32_t)x;
    ++head;
    r.head.store(head, std::memory_order_release);
    return true;
  }

  void mark_run(int t, uint32_t dep) {
    for (int p : producers[dep])
      if (done_epoch[p].load(std::memory_order_acquire) != epoch)
        order_violations.fetch_add(1);
    runs[t].fetch_add(1);
    tasks_run.fetch_add(1);
  }
  void mark_done(int t) {
    done_epoch[t].store(epoch, std::memory_order_release);
  }

  // the device trigger, step for step
  void trigger(int e, const EventDesc& ed0, const int32_t* fan) {
    if (ed0.flags & EV_FAN_CACHED) {
      bool fire = ed0.count == 1;
      if (!fire) fire = counters[e].fetch_add(1u) + 1u == epoch * ed0.count;
      if (fire) {
        // the empty tasks of `e` run here: mark them like the device's
        // inline execution would
        const int n_in = (int)(ed0.flags >> kEvInlineShift);
        for (int t = ed0.last - n_in + 1; t <= ed0.last; ++t) {
          mark_run(t, (uint32_t)g->h_tasks[t].dep);
          mark_done(t);
        }
        counters[fan[0]].fetch_add(1u, std::memory_order_release);
        if (fan[1] >= 0) counters[fan[1]].fetch_add(1u, std::memory_order_release);
      }
      return;
    }
    std::vector<int> stack{e};
    bool first = true;
    while (!stack.empty()) {
      const int ev = stack.back();
      stack.pop_back();
      const EventDesc ed = first ? ed0 : g->h_events[ev];
      first = false;
      if (!(ed.flags & (EV_HAS_JIT | EV_HAS_INLINE))) {
        counters[ev].fetch_add(1u, std::memory_order_release);
        continue;
      }
      const uint32_t old = counters[ev].fetch_add(1u);
      if (old + 1u != epoch * ed.count) continue;
      if (ed.flags & EV_HAS_JIT)
        if (!push(*sched[ev % S], (uint32_t)ev)) return;
      if (ed.flags & EV_HAS_INLINE) {
        const int n_in = (int)(ed.flags >> kEvInlineShift);
        for (int t = ed.last - n_in + 1; t <= ed.last; ++t) {
          mark_run(t, (uint32_t)g->h_tasks[t].dep);
          mark_done(t);
          stack.push_back(g->h_tasks[t].trig);
        }
      }
    }
  }

  void work(std::mt19937& rng) {
    if (max_delay_us <= 0) return;
    const int us = (int)(rng() % (uint32_t)(max_delay_us + 1));
    const auto until = Clock::now() + std::chrono::microseconds(us);
    while (Clock::now() < until) std::this_thread::yield();
  }

  void worker(int w, uint32_t seed) {
    std::mt19937 rng(seed * 7919u + (uint32_t)w);
    const int a1 = g->h_aot_off[w + 1];
    int ai = g->h_aot_off[w];
    uint32_t jit_head = jit[w]->head.load();
    const EventDesc& end = g->h_events[g->bg.end_lin];
    while (!timed_out()) {
      const bool have_head = ai < a1;
      const AotRec* hr = have_head ? &g->h_aot_rec[ai] : nullptr;
      uint32_t v;
      int cmd = -1;
      TaskDesc desc{};
      EventDesc tev{};
      int32_t fan[2] = {-1, -1};
      if (try_pop(*jit[w], jit_head, v)) {
        cmd = (int)v;
        desc = g->h_tasks[cmd];
        tev = g->h_events[desc.trig];
      } else if (have_head && event_done(hr->desc.dep, hr->dep_count)) {
        cmd = hr->id;
        desc = hr->desc;
        tev = hr->trig_ev;
        fan[0] = hr->fan[0];
        fan[1] = hr->fan[1];
        ++ai;
      } else if (!have_head && event_done(g->bg.end_lin, end.count)) {
        break;
      } else {
        std::this_thread::yield();
        continue;
      }
      mark_run(cmd, (uint32_t)desc.dep);
      work(rng);
      mark_done(cmd);
      trigger(desc.trig, tev, fan);
    }
  }

  void scheduler(int s) {
    uint32_t head = sched[s]->head.load();
    uint32_t cursor = (uint32_t)(((int64_t)s * W) / S);
    const EventDesc& end = g->h_events[g->bg.end_lin];
    while (!timed_out()) {
      uint32_t v;
      if (!try_pop(*sched[s], head, v)) {
        if (event_done(g->bg.end_lin, end.count)) break;
        std::this_thread::yield();
        continue;
      }
      const EventDesc ed = g->h_events[v];
      const int n = ed.last - ed.first + 1;
      for (int i = 0; i < n; ++i) {
        const int t = ed.first + i;
        if (g->h_tasks[t].launch != MPK_LAUNCH_JIT) continue;
        const int w = (int)((cursor + (uint32_t)i) % (uint32_t)W);
        if (!push(*jit[w], (uint32_t)t)) return;
      }
      cursor += (uint32_t)n;
    }
  }
};

}  // namespace

extern "C" mpk_status mpk_debug_simulate(const mpk_graph* g, int steps,
                                         uint32_t seed, int max_delay_us,
                                         int timeout_ms, mpk_sim_report* rep) {
  if (!g || !rep || steps < 1 || timeout_ms < 1 || !g->encoded)
    return MPK_ERR_INVALID_ARG;
  std::memset(rep, 0, sizeof(*rep));
  Sim sim(g, max_delay_us);
  const auto t0 = Clock::now();
  for (int step = 1; step <= steps && !sim.abort.load(); ++step) {
    sim.epoch = (uint32_t)step;
    for (auto& r : sim.runs) r.store(0);
    sim.deadline = Clock::now() + std::chrono::milliseconds(timeout_ms);
    // the root event has no producers: it is done at every epoch
    {
      std::vector<std::thread> th;
      for (int s = 0; s < sim.S; ++s) th.emplace_back([&sim, s] { sim.scheduler(s); });
      for (int w = 0; w < sim.W; ++w)
        th.emplace_back([&sim, w, seed, step] { sim.worker(w, seed + (uint32_t)step); });
      for (auto& t : th) t.join();
    }
    if (sim.abort.load()) {
      rep->deadlocked = 1;
      break;
    }
    for (int t = 0; t < sim.nT; ++t) {
      const int r = sim.runs[t].load();
      if (r == 0) ++rep->missing_runs;
      if (r > 1) rep->duplicate_runs += r - 1;
    }
    rep->steps_completed = step;
  }
  rep->tasks_run = sim.tasks_run.load();
  rep->order_violations = sim.order_violations.load();
  rep->seconds = std::chrono::duration<double>(Clock::now() - t0).count();
  return MPK_OK;
}
