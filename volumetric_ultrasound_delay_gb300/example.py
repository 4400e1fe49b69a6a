"""Usage example of the Python binding: one plan, one beamform of a 32 x 32-array
volume (64^3 voxels, 32 frames, 9 transmits, 2048 samples) on the GPU.

Run it with ``python -m volumetric_ultrasound_delay_gb300.example`` after
building libdas (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations


def example():
    """Returns y (B x N float32 CUDA tensor) of a random record."""
    import numpy as np
    import torch

    from volumetric_ultrasound_delay_gb300 import das

    # nx, ny, nz, x0, y0, z0, dx, dy, dz (metres)
    grid = (64, 64, 64, -9.6e-3, -9.6e-3, 5e-3, 0.3e-3, 0.3e-3, 0.7e-3)
    # 32 x 32 receivers at 0.3 mm pitch in the z = 0 plane (metres)
    off = (np.arange(32) - 15.5) * 0.3e-3
    rx = np.stack([np.tile(off, 32), np.repeat(off, 32), np.zeros(1024)], axis=1).astype(np.float32)
    with das.Plan(grid, rx, c=1540.0, fs=20e6, t0=0.0, fnum=1.5, dtype="f32",
                  B=32, Q=9, M=1024, K=2048) as plan:           # kernel="auto"
        rf = torch.randn(32, 9, 1024, 2048, device="cuda")     # B x Q x M x K record
        tau = torch.zeros(9, plan.N, device="cuda")             # Q x N transmit delays (s)
        w = torch.ones(9, plan.N, device="cuda")                # Q x N transmit weights
        y = plan.beamform(rf, tau, w)                           # B x N, on the current stream
    return y


if __name__ == "__main__":
    import torch
    y = example()
    torch.cuda.synchronize()
    print(tuple(y.shape), float(y.abs().max()))
