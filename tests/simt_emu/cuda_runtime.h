// Stand-in for the CUDA runtime header under the host emulation (emu.h).
#pragma once
#include "emu.h"
