// Host-side planning helpers shared by the GEMV launches of gemv.cu and
// chain.cu: the device figures a plan needs, and the per-row arithmetic that
// depends on K alone.
#pragma once

namespace w4 {

// Figures of the device a plan is made for.
struct DeviceInfo {
  int dev = -1;           // device ordinal, -1 when planning without one
  int sms = 0;
  int smem_optin = 0;     // largest dynamic shared memory per CTA
  int smem_per_sm = 0;
  int smem_reserved = 0;  // shared memory the system keeps per CTA
};

// The figures of device `dev` (cached; sms == 0 when they cannot be read).
DeviceInfo device_info(int dev);

// The current device and its figures (false when there is none).
bool current_device(int* dev, DeviceInfo* di);

// The current device's figures, or GB300's when planning without a device.
void planning_device(DeviceInfo* di);

// Lane team T, groups per lane NI, groups per lane per chunk CL and chunks
// nch of a row of K codes (K a multiple of 32).  These fix the association
// of every row sum, so they depend on K alone.
void row_shape(int K, int* T, int* NI, int* CL, int* nch);

// Stage geometry of a window of `rb` rows (whole rows, or `cps` chunks of
// each row under split-K).
void tile_geometry(int K, int T, int CL, bool whole, int cps, int rb, int* code_pitch,
                   int* step_pitch, int* step_off, int* tile_bytes);

}  // namespace w4
