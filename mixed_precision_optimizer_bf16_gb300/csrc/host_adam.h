// host_adam.h -- the host half of the ZeRO-Offload step (bf16opt_create_offload):
// AdamW over FP32 master weights and moments kept in host memory, on the
// host's cores ("企业官网建设流程全解析" (cf-1.com), section 3.3: the DeepSpeed
// configuration with offload_optimizer on the CPU; "单机多卡实战：Megatron-
// DeepSpeed训练类BLOOM模型全流程解析", section 6: optimizer offload as a way to
// fit larger models).
//
// Plain portable C++ (no intrinsics): the same FP32 operations, in the same
// order, as the device's fused step -- explicit fused multiply-adds (std::fma,
// one rounding), IEEE square root and division, every other product rounded
// on its own (the library is built with -ffp-contract=off) -- so that, given
// the scalars and the clip coefficient the device computed, the host update
// gives the device's bits.
#pragma once

#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

namespace bf16host {

// Per-group FP32 scalars of one step (computed on the device, copied here).
struct HostGroup {
    float b1, omb1, b2, omb2, eps, decay, step_size, inv_sqrt_bc2;
};

// bf16 = the FP32 value rounded to its upper 16 bits, to nearest, ties to
// even (IEEE 754 round-to-nearest-even on the dropped half); NaN stays a
// quiet NaN.  Branch-free so the loop below vectorises.
inline uint16_t to_bf16(float x) {
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint32_t hi = u >> 16, lo = u & 0xffffu;
    const uint32_t up = (lo > 0x8000u) | ((lo == 0x8000u) & (hi & 1u));
    const bool nan = (u & 0x7fffffffu) > 0x7f800000u;
    return (uint16_t)(nan ? (hi | 0x40u) : hi + up);
}

// One AdamW step over n elements of one parameter group: the accumulated
// gradient acc (times gscale), clipped by c = c_hi + c_lo; p, m, v updated in
// place, bf the bf16 copy of the new master.
inline void adam_range(const float *__restrict__ acc, float *__restrict__ p, float *__restrict__ m,
                       float *__restrict__ v, uint16_t *__restrict__ bf, uint64_t n, float gscale, float c_hi,
                       float c_lo, const HostGroup &G) {
    for (uint64_t i = 0; i < n; ++i) {
        const float e = acc[i] * gscale;
        const float gc = std::fma(e, c_hi, e * c_lo);                  // clipped gradient
        const float m1 = std::fma(G.b1, m[i], G.omb1 * gc);
        const float v1 = std::fma(G.b2, v[i], G.omb2 * gc * gc);
        const float den = std::fma(std::sqrt(v1), G.inv_sqrt_bc2, G.eps);   // sqrt(v_hat) + eps
        const float upd = m1 / den;
        const float delta = std::fma(G.decay, p[i], G.step_size * upd);  // lr wd p + step_size upd
        const float p1 = p[i] - delta;
        p[i] = p1;
        m[i] = m1;
        v[i] = v1;
        bf[i] = to_bf16(p1);
    }
}

// A fixed set of worker threads; run(f) calls f(w, n) on every worker w in
// [0, n) -- the calling thread is worker 0 -- and returns when all are done.
class Pool {
  public:
    explicit Pool(int n) : n_(n < 1 ? 1 : n) {
        for (int w = 1; w < n_; ++w) th_.emplace_back([this, w] { loop(w); });
    }
    ~Pool() {
        {
            std::lock_guard<std::mutex> lk(mu_);
            quit_ = true;
        }
        cv_.notify_all();
        for (auto &t : th_) t.join();
    }
    int size() const { return n_; }
    void run(const std::function<void(int, int)> &f) {
        {
            std::lock_guard<std::mutex> lk(mu_);
            job_ = &f;
            left_ = n_ - 1;
            ++gen_;
        }
        cv_.notify_all();
        f(0, n_);
        std::unique_lock<std::mutex> lk(mu_);
        done_.wait(lk, [this] { return left_ == 0; });
        job_ = nullptr;
    }

  private:
    void loop(int w) {
        uint64_t seen = 0;
        for (;;) {
            const std::function<void(int, int)> *job;
            {
                std::unique_lock<std::mutex> lk(mu_);
                cv_.wait(lk, [&] { return quit_ || gen_ != seen; });
                if (quit_) return;
                seen = gen_;
                job = job_;
            }
            (*job)(w, n_);
            {
                std::lock_guard<std::mutex> lk(mu_);
                if (--left_ == 0) done_.notify_one();
            }
        }
    }
    int n_;
    std::vector<std::thread> th_;
    std::mutex mu_;
    std::condition_variable cv_, done_;
    const std::function<void(int, int)> *job_ = nullptr;
    uint64_t gen_ = 0;
    int left_ = 0;
    bool quit_ = false;
};

}  // namespace bf16host
