// ctl.h -- launch controls shared by host and device code.
#pragma once

namespace os {

// Controls every kernel with a device-side wait receives: where to report a
// wait that gave up, how long a wait may last, and a host-chosen fault to
// inject (tests only).
struct KernelCtl {
    unsigned int* err;             // device status word; bit 0 = a bounded wait gave up
    unsigned long long timeout_ns; // bound on each device-side wait
    int fault;                     // 0: none; 1: see kFaultSkipFirstLoad
};

constexpr unsigned int kErrWaitTimeout = 1u;
// Fault 1 withholds the first piece of data that a bounded wait expects: the
// first CTA of the bulk-copy ring softmax never issues its first copy, and CTA
// 1 of the first TopK cluster never pushes its first list to CTA 0.
constexpr int kFaultSkipFirstLoad = 1;

}  // namespace os
