"""Helpers for the GPU parity tests: move a synthetic case to the device, launch
through the C ABI into NaN-poisoned outputs with a guard tail, and compare."""
import numpy as np
import torch

from fp8_scaled_gemm_sm_gb300 import binding

NAN_BF16 = 0x7FC0
CANARY = 0x5A5A
CANARY_ELEMS = 4096


def lib_ready():
    from fp8_scaled_gemm_sm_gb300 import build

    build.build()
    return binding.lib()


class DeviceCase:
    """A synth.Case on cuda:0 plus a C buffer with a canary tail."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.A = case.A.to(device)
        self.B = case.B.to(device)
        self.sa = None if case.sa is None else case.sa.to(device)
        self.sb = None if case.sb is None else case.sb.to(device)
        self.buf = torch.empty(case.M * case.N + CANARY_ELEMS, dtype=torch.int16, device=device)
        self.C = self.buf[: case.M * case.N].view(case.M, case.N)
        self.buf[case.M * case.N:].fill_(CANARY)

    def poison(self):
        self.C.fill_(NAN_BF16)

    def canary_ok(self):
        tail = self.buf[self.case.M * self.case.N:]
        return bool((tail == CANARY).all().item())

    def launch(self, h, M=None, stream=None):
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        binding.scaled_gemm_launch(
            h, self.A.data_ptr(), self.B.data_ptr(),
            0 if self.sa is None else self.sa.data_ptr(),
            0 if self.sb is None else self.sb.data_ptr(),
            self.C.data_ptr(), self.case.M if M is None else M, s,
        )

    def c_bits(self):
        return self.C.cpu().numpy().view(np.uint16)


def make_plan(case, M_max=None):
    return binding.scaled_gemm_create(case.mode, case.N, case.K, case.M if M_max is None else M_max)
