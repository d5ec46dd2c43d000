// errors.h -- bits of the device error word (read back by dsa_get_error).
#pragma once
namespace dsa {
constexpr int kErrBounds = 1;   // a selected position or page id out of range; access skipped
constexpr int kErrTimeout = 2;  // a pipeline wait gave up after its time limit
constexpr int kErrSpans = 4;    // a capturable plan's update found invalid spans; the plan was emptied
}  // namespace dsa
