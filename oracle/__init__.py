"""CPU oracle for TurboQuant KV-cache quantization and compressed-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` use it.  It shares no code with the CUDA library.

Everything is plain NumPy in float64 (SciPy for the regularized incomplete beta
function and Gamma function), written in the order and notation of the source
("Вечная математика TurboQuant", blog.sergeynikolenko.ru, sections «Шаг 0»,
«Шаг 1», «Шаг 2», «QJL», «Собственно TurboQuant», Theorems 1 and 2).

Parity status of every function is listed in ``oracle/tq_oracle.py``'s header.
"""
from .tq_oracle import *  # noqa: F401,F403
