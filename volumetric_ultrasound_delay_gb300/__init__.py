"""Volumetric delay-and-sum beamforming on one GB300 (sm_103a).

The computation lives in the CUDA C-ABI library ``_lib/libdas.so`` (sources in
``csrc/``, declarations in ``include/das.h``); :mod:`.das` is its thin ctypes
binding and :mod:`.synth` makes seeded synthetic workloads.  ``Plan`` and
``permute`` are loaded on first use, so importing the package (for example to
use :mod:`.synth`) does not need the built library.
"""
__all__ = ["Plan", "permute", "DasError", "synth"]


def __getattr__(name):
    if name in ("Plan", "permute", "DasError", "lib"):
        from . import das
        return getattr(das, name)
    raise AttributeError(name)
