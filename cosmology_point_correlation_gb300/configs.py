"""The five synthetic workloads, by name and size, and a generator for each.

Each workload is a catalogue recipe (point process, N, box, seed) plus the
counting parameters (periodic flag, r_max, number of linear bins). Sizes and
processes follow the benchmark workloads of this library; the catalogues stand
in for the GRAMSCI v2 paper's test mock, DESI DR1 LRG sample and Quijote
halos, none of which are available here.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import catalogues


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    box_mpc: float
    periodic: bool
    r_max_mpc: float
    nbins: int
    process: str                      # "uniform" | "neyman_scott"
    seed: int
    ns: dict = field(default_factory=dict)   # Neyman-Scott parameters

    @property
    def box_lu(self) -> int:
        return catalogues.box_lattice(self.box_mpc)

    @property
    def edges_lu(self) -> np.ndarray:
        return catalogues.linear_edges_lu(self.r_max_mpc, self.nbins)

    def points(self, n: int | None = None, seed: int | None = None) -> np.ndarray:
        """int32 [n][3] lattice coordinates (default: the full workload)."""
        n = self.n if n is None else n
        seed = self.seed if seed is None else seed
        if self.process == "uniform":
            return catalogues.uniform(n, self.box_mpc, seed)
        # keep the cluster density when a smaller n is requested
        scale = n / self.n
        return catalogues.neyman_scott(n, self.box_mpc,
                                       max(1, int(round(self.ns["n_parents"] * scale))),
                                       self.ns["mu"], self.ns["sigma"], seed)


TINY_3PCF = Workload("tiny_3pcf", 2_000, 100.0, True, 20.0, 10, "uniform", 1001)
CLUSTERED_3PCF_D = Workload("clustered_3pcf_data", 200_000, 500.0, True, 30.0, 15,
                            "neyman_scott", 1002, {"n_parents": 4_000, "mu": 50.0, "sigma": 3.0})
CLUSTERED_3PCF_R = Workload("clustered_3pcf_randoms", 200_000, 500.0, True, 30.0, 15,
                            "uniform", 1003)
LARGE_3PCF = Workload("large_3pcf", 2_000_000, 1000.0, True, 40.0, 20, "uniform", 1004)
BAO_3PCF = Workload("bao_3pcf", 2_000_000, 2000.0, False, 150.0, 30, "neyman_scott", 1005,
                    {"n_parents": 20_000, "mu": 100.0, "sigma": 5.0})
PARITY_4PCF = Workload("parity_4pcf", 200_000, 500.0, True, 20.0, 8, "neyman_scott", 1006,
                       {"n_parents": 4_000, "mu": 50.0, "sigma": 3.0})

ALL = {w.name: w for w in (TINY_3PCF, CLUSTERED_3PCF_D, CLUSTERED_3PCF_R, LARGE_3PCF,
                           BAO_3PCF, PARITY_4PCF)}
