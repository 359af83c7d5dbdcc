"""Device-side generation of a synthetic workload (multi-GB K/V never leave the GPU).

Builds ``synth/_libsynth.so`` from ``synth/csrc/synth_gen.cu`` and fills torch
tensors with exactly the bits ``synth.kv_unit`` produces on the host.  Q, the
heavy rows and their positions are generated on the host and uploaded.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth_gen.cu")
_LIB = os.path.join(_HERE, "_libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
            tmp = _LIB + ".%d.tmp" % os.getpid()
            subprocess.check_call([nvcc, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                                   "-gencode", "arch=compute_103a,code=sm_103a",
                                   "-cudart", "static", "-o", tmp, _SRC])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, ll, ci, cf, cu64 = (ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_float,
                                ctypes.c_ulonglong)
        lib.synth_fill_kv.argtypes = [vp, vp, ci, ci, ll, ci, cu64, cu64, cf, vp, ci, cf, vp]
        lib.synth_place_heavy.argtypes = [vp, ci, ci, ci, ll, ci, vp, vp, ci, vp, vp]
        lib.synth_fill_kv.restype = ci
        lib.synth_place_heavy.restype = ci
        _lib = lib
    return _lib


class DeviceWorkload:
    """Q/K/V of a workload resident on a CUDA device, plus the host-side tables."""

    def __init__(self, wl: synth.Workload, device="cuda"):
        import torch
        self.wl = wl
        self.device = torch.device(device)
        self.cu_host = wl.cu_seqlens()
        self.lengths = wl.seq_lengths()
        self.N_tot = int(self.cu_host[-1])
        L, H, d = wl.num_layers, wl.num_kv_heads, wl.head_dim
        self.q_host = synth.q_window(wl)
        self.outliers = synth.outlier_channels(wl)
        self.heavy_pos = synth.heavy_positions(wl)
        self.heavy_vec = synth.heavy_rows(wl, self.q_host) if wl.num_heavy else None
        with torch.cuda.device(self.device):
            self.cu = torch.from_numpy(self.cu_host).to(self.device)
            self.q = torch.from_numpy(self.q_host.view(np.int16)).to(self.device).view(torch.bfloat16)
            self.k = torch.empty((L, H, self.N_tot, d), dtype=torch.bfloat16, device=self.device)
            self.v = torch.empty_like(self.k)
            stream = torch.cuda.current_stream(self.device)
            oc = torch.from_numpy(np.ascontiguousarray(self.outliers, dtype=np.int32)
                                  .reshape(-1)).to(self.device)
            lib = _load()
            rc = lib.synth_fill_kv(self.k.data_ptr(), self.v.data_ptr(), L, H, self.N_tot, d,
                                   synth.stream_key(wl.seed, synth.S_K),
                                   synth.stream_key(wl.seed, synth.S_V), float(wl.sigma_kv),
                                   oc.data_ptr() if oc.numel() else None, wl.num_outliers,
                                   float(wl.outlier_scale), ctypes.c_void_p(stream.cuda_stream))
            if rc != 0:
                raise RuntimeError("synth_fill_kv failed with CUDA error %d" % rc)
            if wl.num_heavy:
                pos = torch.from_numpy(np.ascontiguousarray(self.heavy_pos, dtype=np.int32)
                                       .reshape(-1)).to(self.device)
                rows = torch.from_numpy(np.ascontiguousarray(self.heavy_vec).view(np.int16)
                                        .reshape(-1)).to(self.device)
                rc = lib.synth_place_heavy(self.k.data_ptr(), wl.num_requests, L, H, self.N_tot, d,
                                           self.cu.data_ptr(), pos.data_ptr(), wl.num_heavy,
                                           rows.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
                if rc != 0:
                    raise RuntimeError("synth_place_heavy failed with CUDA error %d" % rc)
            torch.cuda.synchronize(self.device)

    def unit_host(self, r: int, l: int, h: int):
        """(q_rows [G*w][d], k [n][d], v [n][d]) of one unit as host bf16 bits, regenerated
        on the host from the seed (never read back from the device)."""
        wl = self.wl
        G, w = wl.group, wl.window
        q = self.q_host[r, l, h * G:(h + 1) * G].reshape(G * w, wl.head_dim)
        k, v = synth.kv_unit(wl, r, l, h, outl=self.outliers, heavy_pos=self.heavy_pos,
                             heavy_vec=self.heavy_vec)
        return q, k, v
